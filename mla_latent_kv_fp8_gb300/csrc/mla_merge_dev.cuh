// mla_merge_dev.cuh -- device side of the log-sum-exp merge of partial answers,
// used by the merge kernels (mla_merge.cu): one function per work item, so a
// kernel can map items to warps or CTAs as it sees fit.
//
// "Kimi K3 on AMD Instinct MI355X" post, section 1 (DCP paragraph): each
// partial answer over a part of the history carries normalisation information
// so that the merge weighs the parts correctly.  With lse_s the natural-log
// normaliser of part s:
//     lse = M + ln sum_s exp(lse_s - M),   M = max_s lse_s
//     out = sum_s exp(lse_s - lse) * o_s
// Parts with lse_s = -inf weigh exactly 0; their outputs (never written for an
// empty part) are selected away, never multiplied.
#pragma once

#include <cuda_bf16.h>

#include "mla_internal.cuh"

namespace mla {
namespace mergedev {

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

// Parts of `row` that hold an answer: all p.S of them, or in a decode's split
// combine only the partitions that the row's request reaches (its length read
// and checked as the decode kernels do).
__device__ __forceinline__ int live_parts(const MergeParams& p, int64_t row) {
    if (!p.seq_lens) return p.S;
    int L = __ldg(p.seq_lens + row / p.rows_per_req);
    if (L < 0 || L > p.max_pages * kPage || (L > 0 && L < p.T)) L = 0;
    const int pages = (L + kPage - 1) / kPage;
    const int n = (pages + p.chunk_pages - 1) / p.chunk_pages;
    return n < p.S ? n : p.S;
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

// Few parts (S <= 32): one warp merges (row, 64 value dims chunk); lane s holds
// lse_s, each lane owns two dims.  The normalisers and every part's two
// values are loaded in a single round, so the merge costs one memory latency.
template <bool kBf16In>
__device__ __forceinline__ void merge_warp(const MergeParams& p, int64_t row, int chunk, int lane) {
    const int64_t col = (int64_t)chunk * 64 + lane * 2;
    const int live = live_parts(p, row);  // loaded beside the normalisers, not before them
    float ls = (lane < p.S) ? p.part_lse[(int64_t)lane * p.rows + row] : -INFINITY;
    float2 v[32];
#pragma unroll
    for (int s = 0; s < 32; ++s)
        v[s] = s < p.S ? load2<kBf16In>(p.part_out, ((int64_t)s * p.rows + row) * kDv + col) : make_float2(0.f, 0.f);
    if (lane >= live) ls = -INFINITY;
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
    float2 acc = make_float2(0.f, 0.f);
#pragma unroll
    for (int s = 0; s < 32; ++s) {
        const float ws = __shfl_sync(0xffffffffu, w, s);
        if (ws != 0.f) {
            acc.x = fmaf(ws, v[s].x, acc.x);
            acc.y = fmaf(ws, v[s].y, acc.y);
        }
    }
    __nv_bfloat162 o = __floats2bfloat162_rn(acc.x, acc.y);
    *reinterpret_cast<uint32_t*>(dst) = *reinterpret_cast<uint32_t*>(&o);
    if (chunk == 0 && lane == 0 && p.lse) p.lse[row] = M + logf(sum);
}

// Many rows (a DCP merge, or the split combine of a large batch): one warp
// merges one whole row; lane s holds lse_s (S <= 32) and each lane owns 16
// consecutive value dims, so every part of the row is read with 16-byte loads
// (2 per part in bf16, 4 in fp32).  Parts are loaded four at a time, all loads
// of a round in flight together, and the first round is requested with the
// normalisers, so that a merge of up to four parts costs one memory latency.
// A part of weight 0 is never multiplied, and after the first round not
// loaded either.  Four parts per round take 80 registers in bf16 (three CTAs
// of 256 threads per SM) and 128 in fp32 (two per SM).  Measured on 3,072
// rows: loading the first round only after the weights were known took 7.9
// instead of 5.7 us for 3 fp32 parts; eight bf16 parts per round at two CTAs
// per SM were about a quarter slower on 8 parts.
template <bool kBf16In>
__device__ __forceinline__ void unpack16(const uint4 (&v)[kBf16In ? 2 : 4], float (&x)[16]) {
    if constexpr (kBf16In) {
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const uint32_t w[4] = {v[k].x, v[k].y, v[k].z, v[k].w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                x[8 * k + 2 * j] = __uint_as_float(w[j] << 16);
                x[8 * k + 2 * j + 1] = __uint_as_float(w[j] & 0xffff0000u);
            }
        }
    } else {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            x[4 * k] = __uint_as_float(v[k].x);
            x[4 * k + 1] = __uint_as_float(v[k].y);
            x[4 * k + 2] = __uint_as_float(v[k].z);
            x[4 * k + 3] = __uint_as_float(v[k].w);
        }
    }
}

template <bool kBf16In>
__device__ __forceinline__ void merge_row(const MergeParams& p, int64_t row, int lane) {
    constexpr int kVecs = kBf16In ? 2 : 4;   // 16-byte loads per part and lane
    constexpr int kR = 4;                    // parts per round
    const size_t elem = kBf16In ? 2 : 4;
    const char* base = static_cast<const char*>(p.part_out) + (row * kDv + 16 * lane) * elem;
    const size_t part_stride = static_cast<size_t>(p.rows) * kDv * elem;
    auto load_part = [&](int s, uint4 (&v)[kVecs]) {
        const uint4* src = reinterpret_cast<const uint4*>(base + s * part_stride);
#pragma unroll
        for (int k = 0; k < kVecs; ++k) v[k] = __ldg(src + k);
    };
    // The first round's values are requested together with the normalisers,
    // before the weights are known (every part s < S lies inside the buffer);
    // a part of weight 0 among them is loaded but never multiplied.
    const int live = live_parts(p, row);  // loaded beside the normalisers, not before them
    float ls = (lane < p.S) ? p.part_lse[(int64_t)lane * p.rows + row] : -INFINITY;
    uint4 v[kR][kVecs];
#pragma unroll
    for (int j = 0; j < kR; ++j)
        if (j < p.S) load_part(j, v[j]);
    if (lane >= live) ls = -INFINITY;
    const float M = warp_max(ls);
    uint4* dst = reinterpret_cast<uint4*>(p.out + row * kDv + 16 * lane);
    if (M == -INFINITY) {
        dst[0] = dst[1] = make_uint4(0u, 0u, 0u, 0u);
        if (lane == 0 && p.lse) p.lse[row] = -INFINITY;
        return;
    }
    const float e = (ls == -INFINITY) ? 0.f : exp2f((ls - M) * kLog2e);
    const float sum = warp_sum(e);
    const float w = e / sum;  // lanes >= S: 0
    float acc[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) acc[j] = 0.f;
    for (int s0 = 0;;) {
        float ws[kR];
#pragma unroll
        for (int j = 0; j < kR; ++j) {
            ws[j] = __shfl_sync(0xffffffffu, w, (s0 + j) & 31);
            if (s0 + j >= p.S) ws[j] = 0.f;
        }
#pragma unroll
        for (int j = 0; j < kR; ++j) {
            if (ws[j] != 0.f) {  // warp-uniform
                float x[16];
                unpack16<kBf16In>(v[j], x);
#pragma unroll
                for (int d = 0; d < 16; ++d) acc[d] = fmaf(ws[j], x[d], acc[d]);
            }
        }
        s0 += kR;
        if (s0 >= p.S) break;
        // later rounds: only parts of nonzero weight are loaded
#pragma unroll
        for (int j = 0; j < kR; ++j) {
            const int s = s0 + j;
            const float wj = __shfl_sync(0xffffffffu, w, s & 31);
            if (s < p.S && wj != 0.f) load_part(s, v[j]);
        }
    }
    uint32_t o[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        __nv_bfloat162 h = __floats2bfloat162_rn(acc[2 * j], acc[2 * j + 1]);
        o[j] = *reinterpret_cast<uint32_t*>(&h);
    }
    dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
    dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
    if (lane == 0 && p.lse) p.lse[row] = M + logf(sum);
}

struct CtaScratch {             // shared memory of merge_cta
    float m[8];                 // per warp: maximum normaliser of its parts
    float l[8];                 // per warp: sum of exp(lse_s - m) over its parts
    float part[8][32];          // per warp and dim: sum of exp(lse_s - m) * o_s
};

// Many parts (S > 32): 256 threads (eight warps) merge (row, 32 value dims).
// Warp w takes parts w, w + 8, w + 16, ...; each lane owns one dim.  A warp
// loads 32 of its parts' normalisers (one per lane) together with their values,
// so a round costs one memory latency, and merges them against its own
// maximum; parts beyond 256 take further rounds, folded in by rescaling.  The
// eight warps' results meet once in shared memory (one `sync`).
template <bool kBf16In, class Sync>
__device__ __forceinline__ void merge_cta(const MergeParams& p, int64_t row, int chunk, int tid, CtaScratch& sh,
                                          Sync sync) {
    const int lane = tid & 31, wid = tid >> 5;
    const int col = chunk * 32 + lane;
    float m_w = -INFINITY, l_w = 0.f, acc = 0.f;
    const int live = live_parts(p, row);
    for (int base = 0; base < p.S; base += 256) {
        float v[32];
#pragma unroll
        for (int k = 0; k < 32; ++k) {
            const int s = base + wid + 8 * k;
            v[k] = s < p.S ? load1<kBf16In>(p.part_out, ((int64_t)s * p.rows + row) * kDv + col) : 0.f;
        }
        const int sl = base + wid + 8 * lane;  // this lane's part for the normalisers
        float ls = sl < p.S ? p.part_lse[(int64_t)sl * p.rows + row] : -INFINITY;
        if (sl >= live) ls = -INFINITY;
        const float mr = warp_max(ls);
        if (mr == -INFINITY) continue;  // warp-uniform: no part of this round counts
        const float mn = fmaxf(m_w, mr);
        const float a = (m_w == -INFINITY) ? 0.f : exp2f((m_w - mn) * kLog2e);
        const float e = (ls == -INFINITY) ? 0.f : exp2f((ls - mn) * kLog2e);
        float r = 0.f;
#pragma unroll
        for (int k = 0; k < 32; ++k) {
            const float ek = __shfl_sync(0xffffffffu, e, k);
            if (ek != 0.f) r = fmaf(ek, v[k], r);  // a part of weight 0 is never multiplied
        }
        acc = fmaf(acc, a, r);
        l_w = fmaf(l_w, a, warp_sum(e));
        m_w = mn;
    }
    if (lane == 0) {
        sh.m[wid] = m_w;
        sh.l[wid] = l_w;
    }
    sh.part[wid][lane] = acc;
    sync();
    if (wid == 0) {
        float M = sh.m[0];
#pragma unroll
        for (int i = 1; i < 8; ++i) M = fmaxf(M, sh.m[i]);
        if (M == -INFINITY) {
            p.out[row * kDv + col] = 0;
            if (chunk == 0 && lane == 0 && p.lse) p.lse[row] = -INFINITY;
            return;
        }
        float sum = 0.f, t = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float f = (sh.m[i] == -INFINITY) ? 0.f : exp2f((sh.m[i] - M) * kLog2e);
            sum = fmaf(sh.l[i], f, sum);
            t = fmaf(sh.part[i][lane], f, t);
        }
        __nv_bfloat16 o = __float2bfloat16_rn(t / sum);
        p.out[row * kDv + col] = *reinterpret_cast<uint16_t*>(&o);
        if (chunk == 0 && lane == 0 && p.lse) p.lse[row] = M + logf(sum);
    }
}

}  // namespace mergedev
}  // namespace mla
