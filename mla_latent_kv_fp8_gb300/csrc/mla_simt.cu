// mla_simt.cu -- CUDA-core split-KV MLA decode over a paged FP8 latent cache.
//
// The plain path: FP32 FMAs and warp shuffles, no tensor cores.  It handles
// every supported shape and is the baseline the tcgen05 kernel is measured
// against.  One CTA owns (history partition, request, group of <= 16 rows),
// where a row is one (query position t, head h).  Per 64-position page:
//   1. the page's 36,864 codes are loaded with 16-byte loads (prefetched one
//      page ahead in registers) and widened exactly to f16 in shared memory;
//   2. QK: each thread computes full 576-dim dot products for one position and
//      four rows, in the log2 domain with kv_scale * sm_scale * log2(e) folded;
//   3. online softmax per row (warp max / sum), rescaling the running output;
//   4. PV: each thread owns two value dims for all rows of the group.
// Method: "Kimi K3 on AMD Instinct MI355X" post, section 4 (history split into
// parallel partitions inside one GPU, results combined) and section 1 (each
// partial answer carries its log-sum-exp so partials merge exactly).
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "mla_internal.cuh"

namespace mla {
namespace {

constexpr int kThreads = 256;
constexpr int kRG = 16;                        // rows per CTA
constexpr int kWords = kDqk / 2;               // 288 f16x2 words per position
constexpr int kXStride = kPage + 1;            // [word][position], conflict-free both ways
constexpr int kPStride = kRG + 4;              // [position][row], 16-byte aligned rows
constexpr int kChunks = kPage * kDqk / 16;     // 2304 16-byte chunks per page
constexpr int kChunksPerThread = kChunks / kThreads;  // 9
static_assert(kChunks % kThreads == 0, "page must split evenly over the CTA");

struct Smem {
    uint32_t xs[kWords * kXStride];  // f16x2 code values
    uint32_t qs[kRG * kWords];       // bf16x2 query words [row][word]
    float ps[kPage * kPStride];      // scores, then probabilities
    float m[kRG], l[kRG], alpha[kRG];
    int rowlim[kRG];                 // visible prefix per row; -1 for padding rows
};

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ float2 f16x2_to_float2(uint32_t w) {
    __half2 h = *reinterpret_cast<__half2*>(&w);
    return __half22float2(h);
}

// Two E4M3FN codes (low byte first) -> f16x2; exact for every finite code.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two_codes) {
    __half2_raw r = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(two_codes),
                                               __NV_E4M3);
    return static_cast<uint32_t>(r.x) | (static_cast<uint32_t>(r.y) << 16);
}

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

__device__ __forceinline__ void load_page(const DecodeParams& p, int b, int pg, int tid,
                                          uint4 (&regs)[kChunksPerThread], bool& bad) {
    int32_t pid = __ldg(p.block_table + (int64_t)b * p.bt_stride + pg);
    bad = pid < 0 || pid >= p.num_pages;
    if (bad) {
        if (tid == 0) atomicCAS(p.err, 0, kErrPageRange);
        pid = 0;
    }
    const uint8_t* base = p.kv + (int64_t)pid * (kPage * kDqk);
    const int pos = tid % kPage;
    const int c0 = tid / kPage;
#pragma unroll
    for (int j = 0; j < kChunksPerThread; ++j) {
        const int c = c0 + 4 * j;
        regs[j] = __ldg(reinterpret_cast<const uint4*>(base + pos * kDqk + c * 16));
    }
}

// Rows at or beyond `valid_rows` (past the partition's end, or the whole page
// when its id is out of range) are stored as zeros: their probabilities are 0,
// and zero values keep unread bytes (possibly NaN codes) out of the PV sums.
__device__ __forceinline__ void store_page(Smem& S, int tid, const uint4 (&regs)[kChunksPerThread],
                                           int valid_rows) {
    const int pos = tid % kPage;
    const int c0 = tid / kPage;
    const bool keep = pos < valid_rows;
#pragma unroll
    for (int j = 0; j < kChunksPerThread; ++j) {
        const int c = c0 + 4 * j;
        uint32_t v[4] = {regs[j].x, regs[j].y, regs[j].z, regs[j].w};
        if (!keep) v[0] = v[1] = v[2] = v[3] = 0u;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            S.xs[(8 * c + 2 * k) * kXStride + pos] = e4m3x2_to_f16x2(v[k] & 0xffffu);
            S.xs[(8 * c + 2 * k + 1) * kXStride + pos] = e4m3x2_to_f16x2(v[k] >> 16);
        }
    }
}

__global__ void __launch_bounds__(kThreads, 2) simt_decode_kernel(DecodeParams p) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    Smem& S = *reinterpret_cast<Smem*>(smem_raw);
    const int split = blockIdx.x, b = blockIdx.y, rg0 = blockIdx.z * kRG;
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const int HT = p.H * p.T;

    int L = __ldg(p.seq_lens + b);
    if (L < 0 || L > p.max_pages * kPage || (L > 0 && L < p.T)) {
        if (tid == 0) atomicCAS(p.err, 0, kErrSeqRange);
        L = 0;
    }
    const int p_begin = split * p.chunk_pages * kPage;
    const int p_end = min(L, p_begin + p.chunk_pages * kPage);
    const float kv_scale = __ldg(p.kv_scale);
    const float scale2 = kv_scale * p.sm_scale_log2;

    if (tid < kRG) {
        const int r = rg0 + tid;
        S.rowlim[tid] = (r < HT) ? (L == 0 ? 0 : L - p.T + 1 + r / p.H) : -1;
        S.m[tid] = -INFINITY;
        S.l[tid] = 0.f;
    }
    for (int i = tid; i < kRG * kWords; i += kThreads) {
        const int r = rg0 + i / kWords;
        const int w = i % kWords;
        S.qs[i] = (r < HT) ? __ldg(reinterpret_cast<const uint32_t*>(
                                 p.q + ((int64_t)b * HT + r) * kDqk) + w)
                           : 0u;
    }

    float o[kRG][2];
#pragma unroll
    for (int r = 0; r < kRG; ++r) o[r][0] = o[r][1] = 0.f;

    const int pg_begin = p_begin / kPage;
    const int pg_end = (p_end + kPage - 1) / kPage;
    uint4 regs[kChunksPerThread];
    bool bad_next = false;
    if (pg_begin < pg_end) load_page(p, b, pg_begin, tid, regs, bad_next);

    const int qp = tid % kPage;      // QK: position within the page
    const int qr = tid / kPage;      // QK: rows qr, qr+4, qr+8, qr+12

    for (int pg = pg_begin; pg < pg_end; ++pg) {
        const bool bad = bad_next;
        __syncthreads();  // previous page's PV is done with xs / ps
        store_page(S, tid, regs, bad ? 0 : p_end - pg * kPage);
        if (pg + 1 < pg_end) load_page(p, b, pg + 1, tid, regs, bad_next);
        __syncthreads();

        // ---- QK^T for one position and four rows ----
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        const uint32_t* xcol = S.xs + qp;
#pragma unroll 2
        for (int w = 0; w < kWords; w += 4) {
            float2 x[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) x[k] = f16x2_to_float2(xcol[(w + k) * kXStride]);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint4 qv = *reinterpret_cast<const uint4*>(&S.qs[(qr + 4 * i) * kWords + w]);
                float a = acc[i];
                a = fmaf(bf_lo(qv.x), x[0].x, a);
                a = fmaf(bf_hi(qv.x), x[0].y, a);
                a = fmaf(bf_lo(qv.y), x[1].x, a);
                a = fmaf(bf_hi(qv.y), x[1].y, a);
                a = fmaf(bf_lo(qv.z), x[2].x, a);
                a = fmaf(bf_hi(qv.z), x[2].y, a);
                a = fmaf(bf_lo(qv.w), x[3].x, a);
                a = fmaf(bf_hi(qv.w), x[3].y, a);
                acc[i] = a;
            }
        }
        const int pos = pg * kPage + qp;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int rr = qr + 4 * i;
            const bool vis = !bad && pos < p_end && pos < S.rowlim[rr];
            S.ps[qp * kPStride + rr] = vis ? acc[i] * scale2 : -INFINITY;
        }
        __syncthreads();

        // ---- online softmax: warp `wid` owns rows wid and wid + 8 ----
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const int rr = wid + 8 * k;
            const float s0 = S.ps[lane * kPStride + rr];
            const float s1 = S.ps[(lane + 32) * kPStride + rr];
            const float m_old = S.m[rr];
            const float m_new = fmaxf(m_old, warp_max(fmaxf(s0, s1)));
            float e0 = 0.f, e1 = 0.f;
            if (m_new != -INFINITY) {
                e0 = exp2f(s0 - m_new);
                e1 = exp2f(s1 - m_new);
            }
            S.ps[lane * kPStride + rr] = e0;
            S.ps[(lane + 32) * kPStride + rr] = e1;
            const float lt = warp_sum(e0 + e1);
            if (lane == 0) {
                const float a = (m_new == -INFINITY) ? 1.f : exp2f(m_old - m_new);
                S.alpha[rr] = a;
                S.l[rr] = S.l[rr] * a + lt;
                S.m[rr] = m_new;
            }
        }
        __syncthreads();

        // ---- PV: this thread owns value dims 2*tid, 2*tid + 1 ----
#pragma unroll
        for (int r = 0; r < kRG; ++r) {
            const float a = S.alpha[r];
            o[r][0] *= a;
            o[r][1] *= a;
        }
        const uint32_t* xrow = S.xs + tid * kXStride;
#pragma unroll 4
        for (int pp = 0; pp < kPage; ++pp) {
            const float2 x = f16x2_to_float2(xrow[pp]);
            const float4* prow = reinterpret_cast<const float4*>(S.ps + pp * kPStride);
#pragma unroll
            for (int r4 = 0; r4 < kRG / 4; ++r4) {
                const float4 pv = prow[r4];
                o[4 * r4 + 0][0] = fmaf(pv.x, x.x, o[4 * r4 + 0][0]);
                o[4 * r4 + 0][1] = fmaf(pv.x, x.y, o[4 * r4 + 0][1]);
                o[4 * r4 + 1][0] = fmaf(pv.y, x.x, o[4 * r4 + 1][0]);
                o[4 * r4 + 1][1] = fmaf(pv.y, x.y, o[4 * r4 + 1][1]);
                o[4 * r4 + 2][0] = fmaf(pv.z, x.x, o[4 * r4 + 2][0]);
                o[4 * r4 + 2][1] = fmaf(pv.z, x.y, o[4 * r4 + 2][1]);
                o[4 * r4 + 3][0] = fmaf(pv.w, x.x, o[4 * r4 + 3][0]);
                o[4 * r4 + 3][1] = fmaf(pv.w, x.y, o[4 * r4 + 3][1]);
            }
        }
    }
    __syncthreads();

    // ---- epilogue: normalised partial answer and its log-sum-exp ----
    const bool direct = p.n_splits == 1;
#pragma unroll
    for (int r = 0; r < kRG; ++r) {
        const int row = rg0 + r;
        if (row >= HT) break;
        const float l = S.l[r];
        const int64_t grow = (int64_t)b * HT + row;
        if (direct) {
            const float inv = (l > 0.f) ? kv_scale / l : 0.f;
            __nv_bfloat162 v = __floats2bfloat162_rn(o[r][0] * inv, o[r][1] * inv);
            reinterpret_cast<__nv_bfloat162*>(p.out + grow * kDv)[tid] = v;
        } else if (l > 0.f) {
            const float inv = kv_scale / l;
            const int64_t prow = (int64_t)split * p.B * HT + grow;
            reinterpret_cast<float2*>(p.part_out + prow * kDv)[tid] =
                make_float2(o[r][0] * inv, o[r][1] * inv);
        }
    }
    if (tid < kRG && rg0 + tid < HT) {
        const float l = S.l[tid];
        const float lse = (l > 0.f) ? (S.m[tid] + log2f(l)) * kLn2 : -INFINITY;
        const int64_t grow = (int64_t)b * HT + rg0 + tid;
        if (direct) {
            if (p.lse) p.lse[grow] = lse;
        } else {
            p.part_lse[(int64_t)split * p.B * HT + grow] = lse;
        }
    }
}

}  // namespace

cudaError_t launch_simt_decode(const DecodeParams& p, cudaStream_t stream) {
    static int configured_device = -1;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (configured_device != dev) {
        e = cudaFuncSetAttribute(simt_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)sizeof(Smem));
        if (e != cudaSuccess) return e;
        configured_device = dev;
    }
    const int HT = p.H * p.T;
    dim3 grid(p.n_splits, p.B, (HT + kRG - 1) / kRG);
    simt_decode_kernel<<<grid, kThreads, sizeof(Smem), stream>>>(p);
    return cudaGetLastError();
}

}  // namespace mla
