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
    const float ls = (lane < p.S) ? p.part_lse[(int64_t)lane * p.rows + row] : -INFINITY;
    float2 v[32];
#pragma unroll
    for (int s = 0; s < 32; ++s)
        v[s] = s < p.S ? load2<kBf16In>(p.part_out, ((int64_t)s * p.rows + row) * kDv + col) : make_float2(0.f, 0.f);
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

// Normalisers of up to kSmemParts parts are kept in shared memory; beyond that
// they are re-read from global memory (a slow path for very many parts).
constexpr int kSmemParts = 1024;
constexpr int kFirstRound = 32;  // parts per warp whose values load with the normalisers

struct CtaScratch {             // shared memory of merge_cta
    float lse[kSmemParts];
    float red[8];
    float part[8][32];
};

// Many parts (S > 32): 256 threads (eight warps, synchronised by `sync`) merge
// (row, 32 value dims chunk); the warps split the parts, each lane owns one
// dim; the values of the first 256 parts load in the same round as the
// normalisers, and the warps' sums meet in shared memory.  Every thread of the
// eight warps takes the same path.
template <bool kBf16In, class Sync>
__device__ __forceinline__ void merge_cta(const MergeParams& p, int64_t row, int chunk, int tid, CtaScratch& sh,
                                          Sync sync) {
    const int lane = tid & 31, wid = tid >> 5;
    const int col = chunk * 32 + lane;
    auto lse_at = [&](int s) { return s < kSmemParts ? sh.lse[s] : p.part_lse[(int64_t)s * p.rows + row]; };

    float v[kFirstRound];
#pragma unroll
    for (int k = 0; k < kFirstRound; ++k) {
        const int s = wid + 8 * k;
        v[k] = s < p.S ? load1<kBf16In>(p.part_out, ((int64_t)s * p.rows + row) * kDv + col) : 0.f;
    }
    sync();  // the previous use of the scratch is over
    float mx = -INFINITY;
    for (int s = tid; s < p.S; s += 256) {
        const float l = p.part_lse[(int64_t)s * p.rows + row];
        if (s < kSmemParts) sh.lse[s] = l;
        mx = fmaxf(mx, l);
    }
    mx = warp_max(mx);
    if (lane == 0) sh.red[wid] = mx;
    sync();
    float M = sh.red[0];
#pragma unroll
    for (int i = 1; i < 8; ++i) M = fmaxf(M, sh.red[i]);
    sync();
    if (M == -INFINITY) {
        if (wid == 0) {
            p.out[row * kDv + col] = 0;
            if (chunk == 0 && lane == 0 && p.lse) p.lse[row] = -INFINITY;
        }
        return;
    }
    float sm = 0.f;
    for (int s = tid; s < p.S; s += 256) {
        const float ls = lse_at(s);
        if (ls != -INFINITY) sm += exp2f((ls - M) * kLog2e);
    }
    sm = warp_sum(sm);
    if (lane == 0) sh.red[wid] = sm;
    sync();
    float sum = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) sum += sh.red[i];
    const float lse_out = M + logf(sum);

    float acc = 0.f;
#pragma unroll
    for (int k = 0; k < kFirstRound; ++k) {
        const int s = wid + 8 * k;
        if (s < p.S) {
            const float ls = lse_at(s);
            if (ls != -INFINITY) acc = fmaf(exp2f((ls - lse_out) * kLog2e), v[k], acc);
        }
    }
    for (int s = wid + 8 * kFirstRound; s < p.S; s += 8) {  // beyond 256 parts
        const float ls = lse_at(s);
        if (ls != -INFINITY)
            acc = fmaf(exp2f((ls - lse_out) * kLog2e), load1<kBf16In>(p.part_out, ((int64_t)s * p.rows + row) * kDv + col),
                       acc);
    }
    sh.part[wid][lane] = acc;
    sync();
    if (wid == 0) {
        float t = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) t += sh.part[i][lane];
        __nv_bfloat16 o = __float2bfloat16_rn(t);
        p.out[row * kDv + col] = *reinterpret_cast<uint16_t*>(&o);
        if (chunk == 0 && lane == 0 && p.lse) p.lse[row] = lse_out;
    }
}

}  // namespace mergedev
}  // namespace mla
