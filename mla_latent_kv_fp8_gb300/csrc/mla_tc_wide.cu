// mla_tc_wide.cu -- tcgen05 split-KV MLA decode for units of 17..128 query rows
// (many heads and/or several draft positions), for sm_103a (GB300).
//
// Method: "Kimi K3 on AMD Instinct MI355X" post -- section 4 (history cut into
// parallel partitions whose results are combined), section 1 (multi-token
// verify through the DCP path; partial answers carry their log-sum-exp),
// benchmark section (FP8 KV).
//
// Why a second kernel.  With many rows per request (96 heads, or 12 heads x 4
// draft positions) the attention is a real dense contraction: per page every
// row needs 576 + 512 multiply-adds per position.  Giving each CTA only 16 rows
// (the 12-head kernel's shape) makes every CTA stream its own copy of each page
// and makes the tensor core re-read each page operand from shared memory once
// per 16 rows.  Here one CTA takes up to 64 rows of a (partition, request) unit:
//   * QK^T, swap-AB as in the 12-head kernel: D[64 pos x 2R] = K_page[64 x 576] .
//     [q1 | q2]^T with the exact two-term e4m3 split of the query
//     (q * 2^e = q1 + q2 / 16), R = 32 or 64 padded rows (N = 64 or 128).
//   * The two attention warpgroups split the ROWS, not the pages: warpgroup g
//     owns rows [R/2 g, R/2 (g + 1)) of every page, so each row keeps one
//     reference, one normaliser and one output column set, and no merge of the
//     warpgroups is needed at the end.
//   * PV with the probability split along K: P = p1 + p2 with p1 = e4m3(P) and
//     p2 = e4m3(P - p1).  Both terms multiply the same value tile, so one
//     accumulator D[128 dims x R] per 128-dim block takes K = 128 (64 positions
//     of p1, then the same 64 positions of p2); the output tile needs 4R TMEM
//     columns instead of 8R.  TMEM: 2 score buffers x 2R + 4R = 8R columns.
//   * Per element P - (p1 + p2) is at most max(P 2^-8, 2^-10), with P in
//     (0, 256] and the normaliser (summed in fp32 from the unquantised P) at
//     least 16, so the output keeps the bf16 level of accuracy.
// Warp roles (384 threads, one CTA per SM): warp 0 TMA producer (ring of 3 or 4
// pages), warp 1 issues QK^T, warp 2 issues PV, warp 3 allocates TMEM, warps
// 4-7 / 8-11 are the two attention warpgroups.  Every wait is bounded; on
// timeout the kernel records an error, drains its copies and MMAs, frees TMEM
// and returns.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include <mutex>

#include "mla_internal.cuh"
#include "mla_tc_ptx.cuh"

namespace mla {
namespace {

constexpr int kWThreads = 384;
constexpr int kWSlotBytes = kPage * kDqk;    // 36,864: one page
constexpr int kWBoxBytes = kPage * 64;       // 4,096: 64 positions x 64 dims
constexpr int kWBoxes = kDqk / 64;           // 9
constexpr float kWHeadroom = 8.f;            // log2 units a score may exceed its row's reference
constexpr float kWShift = 4.f;               // a new reference sits this far below the page max

// Compile-time shape of one instantiation: kRp padded rows per CTA (32 or 64).
template <int kRp>
struct Wide {
    static constexpr int kRh = kRp / 2;              // rows per attention warpgroup
    static constexpr int kRL = kRh / 2;              // rows per lane (one position per lane pair)
    static constexpr int kNqk = 2 * kRp;             // QK^T MMA N: q1 rows | q2 rows
    static constexpr int kStages = kRp == 64 ? 3 : 4;
    static constexpr int kQpBytes = kNqk * kDqk;     // 73,728 or 36,864
    static constexpr int kPpKStride = 8 * kRp;       // bytes between 8-position groups of P
    static constexpr int kPpBytes = kRp * 2 * kPage; // [R rows x 128 K] e4m3
    static constexpr uint32_t kSCols = kNqk;         // one score buffer
    static constexpr uint32_t kOCol0 = 2 * kNqk;     // output tile: 4 blocks of kRp columns
    static constexpr uint32_t kTmemCols = 8 * kRp;   // 256 or 512
    static_assert(kOCol0 + 4 * kRp <= kTmemCols, "TMEM budget");
    static_assert(kRL == 8 || kRL == 16, "a lane stores 8 or 16 probability codes");
};

template <int kRp>
struct WideSmem {
    using W = Wide<kRp>;
    uint8_t slot[W::kStages][kWSlotBytes];   // 1024-aligned page tiles (64-byte swizzle)
    uint8_t qp[W::kQpBytes];                 // [q1 | q2] K-major, no swizzle
    uint8_t pp[2][W::kPpBytes];              // [p1 ; p2] along K, MN-major, no swizzle
    float red_m[2][2][W::kRh][4];            // [group][page parity][row][warp] page maxima
    float red_l[2][W::kRh][4];               // [group][row][warp] normaliser partials
    alignas(16) float row_scale[kRp];        // kv_scale * sm_scale * log2(e) * 2^-e
    alignas(16) int rowlim[kRp];             // visible prefix per row; -1 = padding
    uint64_t full[W::kStages], empty[W::kStages];
    uint64_t s_full[2], s_empty[2];          // score buffers
    uint64_t p_full[2];                      // both groups' probabilities of a page are ready
    uint64_t pv_done[2];                     // PV of a page done (buffer = page parity)
    uint64_t mma_done[2];                    // per MMA-issuing thread: its MMAs drained
    uint32_t tmem_base;
    int abort;
};

// Byte offset of (row n, k) in the probability operand: MN-major, no swizzle,
// core matrices of 8 K-entries x 16 rows (16 bytes).  k < 64 are the p1 codes of
// positions 0..63, k >= 64 the p2 codes of the same positions.  Core matrices
// along the rows are 128 B apart; 8-position groups follow every 8R bytes.
template <int kRp>
__device__ __forceinline__ uint32_t wpp_off(int n, int k) {
    return (n >> 4) * 128 + (n & 15) + (k & 7) * 16 + (k >> 3) * Wide<kRp>::kPpKStride;
}

// Two probabilities -> e4m3 codes of p1 = e4m3(P) and of p2 = e4m3(P - p1),
// through f16 (11 significant bits cover the 8 that p1 + p2 keeps).
__device__ __forceinline__ void split_p_k(float a0, float a1, uint32_t& c1, uint32_t& c2) {
    const __half2 h = __floats2half2_rn(a0, a1);
    const __half2_raw hr = *reinterpret_cast<const __half2_raw*>(&h);
    c1 = static_cast<uint32_t>(__nv_cvt_halfraw2_to_fp8x2(hr, __NV_SATFINITE, __NV_E4M3));
    const __half2_raw br = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(c1), __NV_E4M3);
    const __half2 r = __hsub2(h, *reinterpret_cast<const __half2*>(&br));
    c2 = static_cast<uint32_t>(
        __nv_cvt_halfraw2_to_fp8x2(*reinterpret_cast<const __half2_raw*>(&r), __NV_SATFINITE, __NV_E4M3));
}

// Sum of 32 values per lane across the warp: on return lane l holds the sum
// of value index l over all lanes.
__device__ __forceinline__ float warp_transpose_sum32(float (&v)[32], int lane) {
#pragma unroll
    for (int w = 16, sh = 16; w >= 1; w >>= 1, sh >>= 1) {
        const bool hi = (lane & sh) != 0;
#pragma unroll
        for (int i = 0; i < w; ++i) {
            const float send = hi ? v[i] : v[i + w];
            const float keep = hi ? v[i + w] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, sh);
        }
    }
    return v[0];
}

template <int N>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, uint32_t (&r)[N]);
template <>
__device__ __forceinline__ void tmem_ld_cols<16>(uint32_t taddr, uint32_t (&r)[16]) {
    tmem_ld16(taddr, r);
}
template <>
__device__ __forceinline__ void tmem_ld_cols<32>(uint32_t taddr, uint32_t (&r)[32]) {
    tmem_ld32(taddr, r);
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}
template <int N>
__device__ __forceinline__ void tmem_st_cols(uint32_t taddr, const uint32_t (&r)[N]);
template <>
__device__ __forceinline__ void tmem_st_cols<16>(uint32_t taddr, const uint32_t (&r)[16]) {
    tmem_st16(taddr, r);
}
template <>
__device__ __forceinline__ void tmem_st_cols<32>(uint32_t taddr, const uint32_t (&r)[32]) {
    tmem_st32(taddr, r);
}


template <int kRp>
__global__ void __launch_bounds__(kWThreads, 1)
    tc_wide_kernel(const __grid_constant__ CUtensorMap tmap, const __grid_constant__ CUtensorMap tmap_box,
                   const DecodeParams p) {
    using W = Wide<kRp>;
    constexpr int kStages = W::kStages, kRh = W::kRh, kRL = W::kRL;
    extern __shared__ uint8_t smem_raw[];
    WideSmem<kRp>& S =
        *reinterpret_cast<WideSmem<kRp>*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int HT = p.H * p.T;
    // Programmatic dependent of the previous kernel on the stream: nothing is
    // read before this point.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    // G = p.row_ctas CTAs per (partition, request), adjacent in the grid, CTA r
    // taking rows [r * p.rows_per_cta, ...): they run at the same time, so all
    // but the first read each page from L2.
    const int G = p.row_ctas;
    const int crank = static_cast<int>(blockIdx.x % G);
    const int split = blockIdx.x / G, b = blockIdx.y;
    const int r0 = p.rows_per_cta * crank;
    const int HTc = min(p.rows_per_cta, HT - r0);  // rows of this CTA (<= kRp)
    volatile int* abort = &S.abort;

    // Loads that depend only on the launch indices go out first: the
    // producer's first 64 page ids, and the query rows of warps 1..11.
    constexpr int kQR = (kRp + 10) / 11;  // query rows per staging warp
    const int pg_begin = split * p.chunk_pages;
    const int32_t* bt_cta = p.block_table + (int64_t)b * p.bt_stride + pg_begin;
    int32_t pid_cur = 0, pid_nxt = 0;
    uint4 qv[kQR][3];
    if (warp == 0) {
        if (lane == 0) {
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap_box)) : "memory");
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap)) : "memory");
        }
        pid_cur = pg_begin + lane < p.max_pages ? __ldg(bt_cta + lane) : 0;
        pid_nxt = pg_begin + 32 + lane < p.max_pages ? __ldg(bt_cta + 32 + lane) : 0;
    } else {
#pragma unroll
        for (int rr = 0; rr < kQR; ++rr) {
            const int r = warp - 1 + 11 * rr;
            const uint4* src = reinterpret_cast<const uint4*>(p.q + ((int64_t)b * HT + r0 + r) * kDqk);
#pragma unroll
            for (int k = 0; k < 3; ++k) {
                const int c = lane + 32 * k;  // 16-byte chunk: 8 bf16 values
                qv[rr][k] = (r < HTc && c < kDqk / 8) ? __ldg(src + c) : make_uint4(0, 0, 0, 0);
            }
        }
    }
    int L = __ldg(p.seq_lens + b);
    const float kv_scale = __ldg(p.kv_scale);
    if (L < 0 || L > p.max_pages * kPage || (L > 0 && L < p.T)) {
        if (tid == 0) atomicCAS(p.err, 0, kErrSeqRange);
        L = 0;
    }
    const int p_begin = pg_begin * kPage;
    const int p_end = min(L, p_begin + p.chunk_pages * kPage);
    const int n_pages = p_end > p_begin ? (p_end - p_begin + kPage - 1) / kPage : 0;
    if (n_pages == 0) {
        // No history in this partition: out = 0 / lse = -inf (unsplit) or an
        // empty partial (lse = -inf) that the merge skips.
        const int64_t row0 = (int64_t)b * HT + r0;
        if (p.n_splits == 1) {
            for (int idx = tid; idx < HTc * kDv; idx += kWThreads) p.out[row0 * kDv + idx] = 0;
            if (p.lse)
                for (int idx = tid; idx < HTc; idx += kWThreads) p.lse[row0 + idx] = -INFINITY;
        } else {
            for (int idx = tid; idx < HTc; idx += kWThreads)
                p.part_lse[(int64_t)split * p.B * HT + row0 + idx] = -INFINITY;
        }
        return;
    }

    // ---------------- set-up: barriers, TMEM, query operand ----------------
    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&S.full[s], 1);
            mbar_init(&S.empty[s], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&S.s_full[i], 1);
            mbar_init(&S.s_empty[i], 8);   // every attention warp reads every score tile
            mbar_init(&S.p_full[i], 8);    // every attention warp writes its rows of P
            mbar_init(&S.pv_done[i], 1);
            mbar_init(&S.mma_done[i], 1);
        }
        S.abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    __syncthreads();
    // Page i into slot i % kStages (one thread); the first kStages pages as nine
    // boxes (first bytes in sooner), later ones as one 3-D copy.
    int issued = 0;
    auto issue_page = [&](int i, int32_t pid) {
        const int s = i % kStages;
        if (pid < 0 || pid >= p.num_pages) {
            if (crank == 0) atomicCAS(p.err, 0, kErrPageRange);
            pid = 0;  // load a valid page; the attention warps mask and zero it
        }
        mbar_expect_tx(&S.full[s], kWSlotBytes);
        const uint32_t dst = smem_u32(S.slot[s]);
        if (i < kStages) {
#pragma unroll
            for (int j = 0; j < kWBoxes; ++j)
                tma_load_box(dst + j * kWBoxBytes, &tmap_box, 64 * j, pid * kPage, &S.full[s]);
        } else {
            tma_load_page(dst, &tmap, pid * kPage, &S.full[s]);
        }
    };
    if (warp == 0 && !p.test_stall_copies) {
        const int first = min(kStages, n_pages);
        for (int i = 0; i < first; ++i) {
            const int32_t pid = __shfl_sync(0xffffffffu, pid_cur, i);
            if (lane == 0) issue_page(i, pid);
        }
        issued = first;
        __syncwarp();
    }
    if (warp == 3) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(&S.tmem_base)),
                     "r"(W::kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    // Query rows r = warp - 1 + 11 k (< kRp): exact split q * 2^e = q1 + q2 / 16.
    if (warp > 0) {
#pragma unroll
        for (int rr = 0; rr < kQR; ++rr) {
            const int r = warp - 1 + 11 * rr;
            if (r >= kRp) continue;
            if (r < HTc) {
                const uint4* v = qv[rr];
                float amax = 0.f;
#pragma unroll
                for (int k = 0; k < 3; ++k) {
                    const uint32_t w[4] = {v[k].x, v[k].y, v[k].z, v[k].w};
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        amax = fmaxf(amax, fabsf(__uint_as_float(w[j] << 16)));
                        amax = fmaxf(amax, fabsf(__uint_as_float(w[j] & 0xffff0000u)));
                    }
                }
                amax = warp_max_redux(amax);
                int e = 0;
                if (amax > 0.f && amax < INFINITY) e = max(-100, min(100, ilogbf(448.f / amax)));
                const float sc = ldexpf(1.f, e);
#pragma unroll
                for (int k = 0; k < 3; ++k) {
                    const int c = lane + 32 * k;
                    if (c >= kDqk / 8) break;
                    const uint32_t w[4] = {v[k].x, v[k].y, v[k].z, v[k].w};
                    uint32_t q1[2] = {0, 0}, q2[2] = {0, 0};
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const float x0 = __uint_as_float(w[j] << 16) * sc;
                        const float x1 = __uint_as_float(w[j] & 0xffff0000u) * sc;
                        const uint32_t c1 = f2_to_e4m3x2(x0, x1);
                        const float2 back = e4m3x2_to_f2(c1);
                        const uint32_t c2 = f2_to_e4m3x2((x0 - back.x) * 16.f, (x1 - back.y) * 16.f);
                        q1[j >> 1] |= c1 << (16 * (j & 1));
                        q2[j >> 1] |= c2 << (16 * (j & 1));
                    }
                    const int k0 = 8 * c;
                    *reinterpret_cast<uint2*>(S.qp + kmajor_off(r, k0, kDqk)) = make_uint2(q1[0], q1[1]);
                    *reinterpret_cast<uint2*>(S.qp + kmajor_off(kRp + r, k0, kDqk)) = make_uint2(q2[0], q2[1]);
                }
                if (lane == 0) {
                    S.row_scale[r] = kv_scale * p.sm_scale_log2 * ldexpf(1.f, -e);
                    S.rowlim[r] = (L == 0) ? 0 : L - p.T + 1 + (r0 + r) / p.H;
                }
            } else {
                for (int c = lane; c < kDqk / 8; c += 32) {
                    *reinterpret_cast<uint2*>(S.qp + kmajor_off(r, 8 * c, kDqk)) = make_uint2(0, 0);
                    *reinterpret_cast<uint2*>(S.qp + kmajor_off(kRp + r, 8 * c, kDqk)) = make_uint2(0, 0);
                }
                if (lane == 0) {
                    S.row_scale[r] = 0.f;
                    S.rowlim[r] = -1;
                }
            }
        }
    }
    fence_async_smem();  // query operand: generic writes -> tensor-core reads
    tc_fence_before();
    if (warp > 0) asm volatile("bar.sync 3, %0;" ::"n"(kWThreads - 32) : "memory");  // warps 1..11
    tc_fence_after();
    const uint32_t tmem = warp > 0 ? S.tmem_base : 0u;
    asm volatile("griddepcontrol.launch_dependents;");

    if (warp == 0) {
        // ======================= TMA producer =======================
        if (!p.test_stall_copies) {
            for (int i = issued; i < n_pages; ++i) {
                if ((i & 31) == 0) {  // next window of page ids; prefetch the one after
                    pid_cur = pid_nxt;
                    pid_nxt = i + 32 + lane < n_pages ? __ldg(bt_cta + i + 32 + lane) : 0;
                }
                const int32_t pid = __shfl_sync(0xffffffffu, pid_cur, i & 31);
                if (!warp_wait(&S.empty[i % kStages], ((i / kStages) & 1) ^ 1, abort, p.err)) break;
                if (lane == 0) issue_page(i, pid);
                __syncwarp();
                issued = i + 1;
            }
        }
        if (lane == 0) {
            // never leave with a copy in flight into this CTA's shared memory
            const uint64_t t0 = global_ns();
            for (int i = max(0, issued - kStages); i < issued; ++i) {
                const int s = i % kStages;
                const uint32_t par = (i / kStages) & 1;
                while (!mbar_try_wait(&S.full[s], par) && global_ns() - t0 < kTimeoutNs) {
                }
            }
        }
    } else if (warp == 1) {
        // ======================= QK^T issuer =======================
        // One thread issues all 18 MMAs of a page (each N = 2R wide, long enough
        // to hide the issue cost).  Pages are taken in order, so the parity of
        // a slot's full barrier is exact.
        const bool leader = elect_one();
        const uint64_t qd = smem_desc(smem_u32(S.qp), 128, (kDqk / 16) * 128, kLayoutNone);
        constexpr uint32_t kIdesc = idesc_e4m3(64, W::kNqk, false, false);
        for (int i = 0; i < n_pages; ++i) {
            const int sb = i & 1;
            if (!warp_wait(&S.full[i % kStages], (i / kStages) & 1, abort, p.err)) break;
            if (!warp_wait(&S.s_empty[sb], ((i >> 1) & 1) ^ 1, abort, p.err)) break;
            tc_fence_after();
            const uint64_t ad = smem_desc(smem_u32(S.slot[i % kStages]), 16, 512, kLayoutSw64);
            const uint32_t d = tmem + W::kSCols * sb;
            if (leader) {
#pragma unroll
                for (int ks = 0; ks < kDqk / 32; ++ks)
                    mma_e4m3(d, ad + static_cast<uint64_t>(((ks >> 1) * kWBoxBytes + (ks & 1) * 32) >> 4),
                             qd + static_cast<uint64_t>(ks * 16), kIdesc, ks > 0);
                mma_commit(&S.s_full[sb]);
            }
            __syncwarp();
        }
        if (leader) {
            mma_commit(&S.mma_done[0]);
            const uint64_t t0 = global_ns();
            while (!mbar_try_wait(&S.mma_done[0], 0) && global_ns() - t0 < kTimeoutNs) {
            }
        }
        __syncwarp();
    } else if (warp == 2) {
        // ======================= PV issuer =======================
        // O[128c + dim][row] += sum_k V^T[dim][k] P[k][row] over K = 128: k < 64 the
        // p1 codes, k >= 64 the p2 codes, both against the same value tile.
        const bool leader = elect_one();
        constexpr uint32_t kIdesc = idesc_e4m3(128, kRp, true, true);
        for (int i = 0; i < n_pages; ++i) {
            const int s = i % kStages, kb = i & 1;
            if (!warp_wait(&S.p_full[kb], (i >> 1) & 1, abort, p.err)) break;
            tc_fence_after();
            const uint64_t ad = smem_desc(smem_u32(S.slot[s]), kWBoxBytes, 512, kLayoutSw64);
            // MN-major, no swizzle: LBO = stride between 8-position groups (K),
            // SBO = stride between 16-row core matrices (N).
            const uint64_t bd = smem_desc(smem_u32(S.pp[kb]), W::kPpKStride, 128, kLayoutNone);
            if (leader) {
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
#pragma unroll
                    for (int c = 0; c < kDv / 128; ++c)
                        mma_e4m3(tmem + W::kOCol0 + kRp * c,
                                 ad + static_cast<uint64_t>((2 * c * kWBoxBytes + (ks & 1) * 32 * 64) >> 4),
                                 bd + static_cast<uint64_t>((ks * 4 * W::kPpKStride) >> 4), kIdesc,
                                 i > 0 || ks > 0);
                mma_commit(&S.pv_done[kb]);
                mma_commit(&S.empty[s]);
            }
            __syncwarp();
        }
        if (leader) {
            mma_commit(&S.mma_done[1]);
            const uint64_t t0 = global_ns();
            while (!mbar_try_wait(&S.mma_done[1], 0) && global_ns() - t0 < kTimeoutNs) {
            }
        }
        __syncwarp();
    } else if (warp >= 4) {
        // ======================= attention warpgroups =======================
        // Warpgroup g owns rows [kRh g, kRh (g + 1)) of every page.  In the M = 64
        // score tile a warp's lanes 0..15 hold its 16 positions; lane l < 16 keeps
        // rows 0..kRL-1 of its group for position l and sends rows kRL..kRh-1 to
        // lane l + 16, so every lane works on kRL rows of one position.  A row's
        // probabilities are P = 2^(s - r) against a reference r that moves only
        // when a score would exceed r + kWHeadroom; the accumulated output columns
        // of the moved rows are then rescaled in place in TMEM.
        const int g = (warp - 4) >> 2;
        const int quad = warp & 3;
        const int half = lane >> 4;
        const int pr = 16 * quad + (lane & 15);   // position within the page
        const int d = 32 * quad + lane;           // latent dim within each 128-dim block
        const int grow0 = kRh * g + kRL * half;   // this lane's first row
        const float NEG = -INFINITY;
        const bool causal = p.T > 1;              // for T = 1 the partition end bounds every row
        const uint32_t lane_base = static_cast<uint32_t>(32 * quad) << 16;
        const uint32_t to = tmem + lane_base + W::kOCol0 + kRh * g;  // block 0 of this group's output
        const int32_t* bt = p.block_table + (int64_t)b * p.bt_stride + pg_begin;
        float lp[kRL], rsc[kRL], rr[kRL];
        float r_l = NEG;                          // lane h < kRh: reference of group row h
#pragma unroll
        for (int j = 0; j < kRL; ++j) {
            lp[j] = 0.f;
            rr[j] = NEG;
            rsc[j] = S.row_scale[grow0 + j];
        }
        bool fail = false;
        int32_t pid_next = __ldg(bt);
        for (int i = 0; i < n_pages; ++i) {
            const int sb = i & 1, kb = i & 1;
            const int32_t pid = pid_next;
            if (i + 1 < n_pages) pid_next = __ldg(bt + i + 1);
            const bool page_ok = pid >= 0 && pid < p.num_pages;
            const int pos = (pg_begin + i) * kPage + pr;
            float s[kRL];
            bool over = false;  // a score of this lane exceeds its row's reference + headroom
#pragma unroll
            for (int j = 0; j < kRL; ++j) s[j] = NEG;
            // ---- scores of this page ----
            if (!fail) fail = !warp_wait(&S.s_full[sb], (i >> 1) & 1, abort, p.err);
            if (!fail) {
                tc_fence_after();
                uint32_t r1[kRh], r2[kRh];
                const uint32_t ta = tmem + lane_base + W::kSCols * sb + kRh * g;
                tmem_ld_cols<kRh>(ta, r1);        // q1 . x of the group's rows
                tmem_ld_cols<kRh>(ta + kRp, r2);  // q2 . x
                tmem_wait_ld();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&S.s_empty[sb]);
                const bool in_part = page_ok && pos < p_end;
#pragma unroll
                for (int j = 0; j < kRL; ++j) {
                    const float lo = __uint_as_float(r1[j]) + __uint_as_float(r2[j]) * 0.0625f;
                    const float hi = __uint_as_float(r1[kRL + j]) + __uint_as_float(r2[kRL + j]) * 0.0625f;
                    const float moved = __shfl_xor_sync(0xffffffffu, hi, 16);
                    const float v = (half ? moved : lo) * rsc[j];
                    const int row = grow0 + j;
                    s[j] = (row < HTc && in_part && (!causal || pos < S.rowlim[row])) ? v : NEG;
                    over |= s[j] > rr[j] + kWHeadroom;  // rr = -inf: any score moves it
                }
            }
            // One barrier per page decides whether any row's reference moves; only
            // then are the page maxima reduced (a second barrier).
            if (group_sync_or(g, fail || over)) {
                if (!fail) {
                    float mine = NEG;  // lane 16 half + j (j < kRL): this warp's max of row kRL half + j
#pragma unroll
                    for (int j = 0; j < kRL; ++j) {
                        const float wlo = warp_max_redux(half ? NEG : s[j]);
                        const float whi = warp_max_redux(half ? s[j] : NEG);
                        mine = ((lane & 15) == j) ? (half ? whi : wlo) : mine;
                    }
                    if ((lane & 15) < kRL) S.red_m[g][kb][kRL * half + (lane & 15)][quad] = mine;
                }
                if (group_sync_or(g, fail)) {
                    fail = true;
                    break;
                }
                float t = NEG;
                if (lane < kRh) {
                    const float4 vm = *reinterpret_cast<const float4*>(S.red_m[g][kb][lane]);
                    t = fmaxf(fmaxf(vm.x, vm.y), fmaxf(vm.z, vm.w));
                }
                const bool need = lane < kRh && t > r_l + kWHeadroom;
                if (__ballot_sync(0xffffffffu, need)) {
                    const float rn = need ? t - kWShift : r_l;
                    const float a = need ? exp2f(r_l - rn) : 1.f;  // r_l = -inf: nothing to keep
                    r_l = rn;
#pragma unroll
                    for (int j = 0; j < kRL; ++j) {
                        rr[j] = __shfl_sync(0xffffffffu, rn, kRL * half + j);
                        lp[j] *= __shfl_sync(0xffffffffu, a, kRL * half + j);
                    }
                    if (i > 0) {
                        // The tile holds PV of pages 0..i-1: wait for the last one, then
                        // scale this group's columns (every warp its own lane quadrant).
                        if (!warp_wait(&S.pv_done[(i - 1) & 1], ((i - 1) >> 1) & 1, abort, p.err)) {
                            fail = true;
                        } else {
                            tc_fence_after();
#pragma unroll
                            for (int c = 0; c < 4; ++c) {
                                uint32_t v[kRh];
                                tmem_ld_cols<kRh>(to + kRp * c, v);
                                tmem_wait_ld();
#pragma unroll
                                for (int j = 0; j < kRh; ++j)
                                    v[j] = __float_as_uint(__uint_as_float(v[j]) * __shfl_sync(0xffffffffu, a, j));
                                tmem_st_cols<kRh>(to + kRp * c, v);
                            }
                            tmem_wait_st();
                        }
                    }
                }
            }
            // ---- probabilities of this page -> [p1 ; p2] operand rows of this group ----
            // Buffer kb was last read by the PV of page i - 2.
            if (!fail && i >= 2) fail = !warp_wait(&S.pv_done[kb], ((i - 2) >> 1) & 1, abort, p.err);
            if (!fail) {
                uint32_t w1[kRL / 4], w2[kRL / 4];
#pragma unroll
                for (int j = 0; j < kRL / 4; ++j) w1[j] = w2[j] = 0u;
#pragma unroll
                for (int j = 0; j < kRL; ++j) {
                    s[j] = (s[j] == NEG) ? 0.f : exp2f(s[j] - rr[j]);
                    lp[j] += s[j];
                }
#pragma unroll
                for (int j = 0; j < kRL; j += 2) {
                    uint32_t c1, c2;
                    split_p_k(s[j], s[j + 1], c1, c2);
                    w1[j >> 2] |= (c1 & 0xffffu) << (8 * (j & 3));
                    w2[j >> 2] |= (c2 & 0xffffu) << (8 * (j & 3));
                }
                uint8_t* pp = S.pp[kb];
                if constexpr (kRL == 16) {
                    *reinterpret_cast<uint4*>(pp + wpp_off<kRp>(grow0, pr)) = make_uint4(w1[0], w1[1], w1[2], w1[3]);
                    *reinterpret_cast<uint4*>(pp + wpp_off<kRp>(grow0, kPage + pr)) =
                        make_uint4(w2[0], w2[1], w2[2], w2[3]);
                } else {
                    *reinterpret_cast<uint2*>(pp + wpp_off<kRp>(grow0, pr)) = make_uint2(w1[0], w1[1]);
                    *reinterpret_cast<uint2*>(pp + wpp_off<kRp>(grow0, kPage + pr)) = make_uint2(w2[0], w2[1]);
                }
                // Positions past the partition's end (or of a page whose id was out
                // of range) may hold anything, even NaN codes: zero them so that
                // 0 * x stays 0 in the PV product.  Their QK^T is already done.
                if (g == 0 && half == 0 && (!page_ok || pos >= p_end)) {
                    uint8_t* row = S.slot[i % kStages] + pr * 64;
#pragma unroll
                    for (int j = 0; j < kWBoxes; ++j) {
                        uint4* q4 = reinterpret_cast<uint4*>(row + j * kWBoxBytes);
                        q4[0] = q4[1] = q4[2] = q4[3] = make_uint4(0, 0, 0, 0);
                    }
                }
                fence_async_smem();
                tc_fence_before();  // TMEM stores of a rescale precede the next PV
                __syncwarp();
                if (lane == 0) mbar_arrive(&S.p_full[kb]);
            }
        }

        // ---- this group's rows: normaliser, log-sum-exp, output ----
        bool o_ok = !fail;
        if (o_ok) o_ok = warp_wait(&S.pv_done[(n_pages - 1) & 1], ((n_pages - 1) >> 1) & 1, abort, p.err);
        if constexpr (kRh == 32) {
            float e[32];
#pragma unroll
            for (int h = 0; h < 32; ++h) e[h] = ((h >> 4) == half) ? lp[h & 15] : 0.f;
            S.red_l[g][lane][quad] = warp_transpose_sum32(e, lane);
        } else {
            float e[16];
#pragma unroll
            for (int h = 0; h < 16; ++h) e[h] = ((h >> 3) == half) ? lp[h & 7] : 0.f;
            const float wsum = warp_transpose_reduce<false>(e, lane);
            if ((lane & 1) == 0) S.red_l[g][lane >> 1][quad] = wsum;
        }
        const bool bad = group_sync_or(g, !o_ok);  // partials written; failure anywhere in the group
        float w = 0.f;                            // lane h < kRh: weight of group row h
        if (lane < kRh) {
            const float4 vl = *reinterpret_cast<const float4*>(S.red_l[g][lane]);
            const float l = (vl.x + vl.y) + (vl.z + vl.w);
            w = (l > 0.f && !bad) ? kv_scale / l : 0.f;
            const int row = kRh * g + lane;
            if (quad == 0 && row < HTc) {
                const float lse = (l > 0.f && !bad) ? (r_l + log2f(l)) * kLn2 : -INFINITY;
                const int64_t grow = (int64_t)b * HT + r0 + row;
                if (p.n_splits == 1) {
                    if (p.lse) p.lse[grow] = lse;
                } else {
                    p.part_lse[(int64_t)split * p.B * HT + grow] = lse;
                }
            }
        }
        if (!bad) tc_fence_after();
        const int64_t row0 = (int64_t)b * HT + r0;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            uint32_t v[kRh];
            if (!bad) {
                tmem_ld_cols<kRh>(to + kRp * c, v);
                tmem_wait_ld();
            } else {
#pragma unroll
                for (int j = 0; j < kRh; ++j) v[j] = 0u;
            }
#pragma unroll
            for (int j = 0; j < kRh; ++j) {
                const float wj = __shfl_sync(0xffffffffu, w, j);
                const int row = kRh * g + j;
                if (row < HTc) {
                    const float o = __uint_as_float(v[j]) * wj;
                    const int64_t at = (row0 + row) * kDv + 128 * c + d;
                    if (p.n_splits == 1)
                        p.out[at] = __bfloat16_as_ushort(__float2bfloat16_rn(o));
                    else
                        p.part_out[(int64_t)split * p.B * HT * kDv + at] = o;
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 3) {
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(S.tmem_base),
                     "r"(W::kTmemCols)
                     : "memory");
    }
}
}  // namespace

// Launch the wide kernel for a unit of p.rows_per_cta rows per CTA (<= 64) and
// p.row_ctas CTAs per (partition, request); the maps are those of the
// 12-head kernel (3-D page view and 2-D box view of the cache).
cudaError_t launch_tc_wide(const DecodeParams& p, const CUtensorMap& map, const CUtensorMap& map_box,
                           cudaStream_t stream) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    static bool ready[64];
    static std::mutex mu;
    {
        std::lock_guard<std::mutex> lk(mu);
        if (!ready[dev]) {
            if ((e = cudaFuncSetAttribute(tc_wide_kernel<32>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          (int)sizeof(WideSmem<32>) + 1024)) != cudaSuccess)
                return e;
            if ((e = cudaFuncSetAttribute(tc_wide_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          (int)sizeof(WideSmem<64>) + 1024)) != cudaSuccess)
                return e;
            ready[dev] = true;
        }
    }
    if (p.rows_per_cta < 1 || p.rows_per_cta > 64 || p.row_ctas < 1 ||
        (int64_t)p.rows_per_cta * p.row_ctas < (int64_t)p.H * p.T)
        return cudaErrorInvalidValue;
    const bool narrow = p.rows_per_cta <= 32;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(p.row_ctas) * static_cast<unsigned>(p.n_splits),
                       static_cast<unsigned>(p.B));
    cfg.blockDim = dim3(kWThreads);
    cfg.dynamicSmemBytes = (narrow ? sizeof(WideSmem<32>) : sizeof(WideSmem<64>)) + 1024;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = narrow ? cudaLaunchKernelEx(&cfg, tc_wide_kernel<32>, map, map_box, p)
               : cudaLaunchKernelEx(&cfg, tc_wide_kernel<64>, map, map_box, p);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace mla
