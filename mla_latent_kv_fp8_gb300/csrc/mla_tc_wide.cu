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
// row needs 576 + 512 multiply-adds per position.  The 12-head kernel gives a
// CTA 16 rows, so every 16 rows would stream their own copy of each page and
// make the tensor core re-read each page operand from shared memory.  Here a
// CTA takes 32 rows of a (partition, request) unit, and ceil(rows / 32) CTAs,
// adjacent in the grid, share each page through L2.
//   * QK^T, swap-AB as in the 12-head kernel: D[64 pos x 64] = K_page[64 x 576] .
//     [q1 | q2]^T with the exact two-term e4m3 split of the query
//     (q * 2^e = q1 + q2 / 16).  One thread needs ~40 cycles to issue a
//     tcgen05.mma, so the 18 MMAs of a page are split along K between two
//     warps, each accumulating its half of the dims into its own 64 columns;
//     the attention warps add the halves.
//   * Four attention warpgroups split the ROWS: warpgroup g owns rows
//     [8g, 8g + 8) of every page, so each row keeps one reference, one
//     normaliser and one output column pair, and no merge of warpgroups is
//     needed at the end.  Each lane works on 4 rows of one position.
//   * PV: D[128 dims x 64] += V^T[128 x 64 pos] . [p1 | p2]^T per 128-dim block,
//     P = p1 + p2 / 16 in e4m3 (relative error ~2^-8), 8 MMAs of N = 64 per page.
//     A row's reference moves when a score would exceed it by 8.8 (log2
//     units) and then sits S = p.ref_shift (4..7, from the partition length)
//     below the page max, so the largest probability starts at 2^S and the
//     e4m3 floor of tiny probabilities lies ~2^-(14+S) below it.
//   * TMEM: 2 score tiles x 128 columns + output 4 blocks x 64 columns = 512.
// Warp roles (640 threads, one CTA per SM): warp 0 TMA producer (ring of 4
// pages), warps 1 and 3 issue QK^T, warp 2 issues PV, warps 4-19 are the four
// attention warpgroups.  Every wait is bounded; on timeout the kernel
// records an error, drains its copies and MMAs, frees TMEM and returns.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include <climits>
#include <mutex>

#include "mla_internal.cuh"
#include "mla_tc_ptx.cuh"

namespace mla {
namespace {

constexpr int kWThreads = 640;               // 20 warps
constexpr int kWGroups = 4;                  // attention warpgroups
constexpr int kWRows = 32;                   // rows (t, h) per CTA
constexpr int kWRg = kWRows / kWGroups;      // 8 rows per warpgroup
constexpr int kWRL = kWRg / 2;               // 4 rows per lane
constexpr int kWN = 2 * kWRows;              // MMA N: q1 | q2 rows (QK), p1 | p2 rows (PV)
constexpr int kWStages = 4;                  // page slots in the TMA ring
constexpr int kWSBufs = 2;                   // score tiles in TMEM, each two K-halves of 64 columns
constexpr int kWPBufs = 4;                   // probability operands in shared memory
constexpr int kWSlotBytes = kPage * kDqk;    // 36,864: one page
constexpr int kWBoxBytes = kPage * 64;       // 4,096: 64 positions x 64 dims
constexpr int kWBoxes = kDqk / 64;           // 9
constexpr int kWQpBytes = kWN * kDqk;        // 36,864
constexpr int kWPpKStride = kWN / 16 * 128;  // 512: bytes between 8-position groups of P
constexpr int kWPpBytes = kWN * kPage;       // 4,096
constexpr uint32_t kWTmemCols = 512;
constexpr uint32_t kWSCols = 2 * kWN;        // 128: one score tile (K-half a | K-half b)
constexpr uint32_t kWOCol0 = kWSBufs * kWSCols;  // 256: output tile, block c at + 64 c
constexpr int kWSetupBar = 1 + kWGroups;     // named barrier of the set-up (warps 1..19)
// log2 units a score may exceed its row's reference: P = 2^(s - r) <= 2^8.8 < 448
constexpr float kWHeadroom = 8.8f;
static_assert(kWOCol0 + 4 * kWN <= kWTmemCols, "TMEM budget");
// The probabilities of page i go to buffer i % kWPBufs, last read by the PV of
// page i - kWPBufs.  With as many buffers as ring slots that PV has finished
// before the scores of page i exist (page i was copied into the slot that PV
// released, and QK^T of page i waited for the copy), so no wait is needed;
// with fewer buffers the attention warps wait for it.
static_assert(kWPBufs <= kWStages, "probability buffers");

struct WideSmem {
    uint8_t slot[kWStages][kWSlotBytes];     // 1024-aligned page tiles (64-byte swizzle)
    uint8_t qp[kWQpBytes];                   // [q1 | q2] K-major, no swizzle
    uint8_t pp[kWPBufs][kWPpBytes];          // [p1 | p2] MN-major, no swizzle
    float red_m[kWGroups][2][kWRg][4];       // [group][page parity][row][warp] page maxima
    float red_l[kWGroups][kWRg][4];          // [group][row][warp] normaliser partials
    alignas(16) float row_scale[kWRows];     // kv_scale * sm_scale * log2(e) * 2^-e
    alignas(16) int rowlim[kWRows];          // visible prefix per row; -1 = padding
    uint64_t full[kWStages], empty[kWStages];
    uint64_t s_full[kWSBufs], s_empty[kWSBufs];
    uint64_t p_full[kWPBufs];                // every warpgroup's rows of P for a page are ready
    uint64_t pv_done[kWPBufs];               // PV of a page done
    uint64_t mma_done[3];                    // per MMA-issuing thread: its MMAs drained
    uint32_t tmem_base;
    int abort;
};
static_assert(sizeof(uint8_t[kWStages][kWSlotBytes]) % 1024 == 0, "slots keep 1 KB alignment");

// Byte offset of (column n, position k) in the probability operand: MN-major,
// no swizzle, core matrices of 8 positions x 16 columns (16 bytes).  Columns
// n < 32 are the p1 codes of rows 0..31, n >= 32 the p2 codes; core matrices
// along n are 128 B apart, 8-position groups 512 B.
__device__ __forceinline__ uint32_t wpp_off(int n, int k) {
    return (n >> 4) * 128 + (n & 15) + (k & 7) * 16 + (k >> 3) * kWPpKStride;
}

// Two probabilities -> e4m3 codes of p1 and of 16 * (value - p1), computed in
// f16 (11 significant bits cover the 8 that p1 + p2 / 16 keeps).
__device__ __forceinline__ void wsplit_p(float a0, float a1, uint32_t& c1, uint32_t& c2) {
    const __half2 h = __floats2half2_rn(a0, a1);
    const __half2_raw hr = *reinterpret_cast<const __half2_raw*>(&h);
    c1 = static_cast<uint32_t>(__nv_cvt_halfraw2_to_fp8x2(hr, __NV_SATFINITE, __NV_E4M3));
    const __half2_raw br = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(c1), __NV_E4M3);
    const __half2 r = __hmul2(__hsub2(h, *reinterpret_cast<const __half2*>(&br)), __float2half2_rn(16.f));
    c2 = static_cast<uint32_t>(
        __nv_cvt_halfraw2_to_fp8x2(*reinterpret_cast<const __half2_raw*>(&r), __NV_SATFINITE, __NV_E4M3));
}

// 2^x with the special function unit (inputs here lie in [-inf, 8]).
__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Sum of 8 values per lane across the warp: on return lane l holds the sum of
// value index l >> 2 over all lanes.
__device__ __forceinline__ float warp_transpose_sum8(float (&v)[8], int lane) {
#pragma unroll
    for (int w = 4, sh = 16; w >= 1; w >>= 1, sh >>= 1) {
        const bool hi = (lane & sh) != 0;
#pragma unroll
        for (int i = 0; i < w; ++i) {
            const float send = hi ? v[i] : v[i + w];
            const float keep = hi ? v[i + w] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, sh);
        }
    }
    float s = v[0];
    s += __shfl_xor_sync(0xffffffffu, s, 2);
    s += __shfl_xor_sync(0xffffffffu, s, 1);
    return s;
}

__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t (&r)[8]) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
                   "=r"(r[7])
                 : "r"(taddr));
}
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&r)[8]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr),
                 "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
                 : "memory");
}


template <bool kLpt>
__global__ void __launch_bounds__(kWThreads, 1)
    tc_wide_kernel(const __grid_constant__ CUtensorMap tmap, const __grid_constant__ CUtensorMap tmap_box,
                   const DecodeParams p) {
    extern __shared__ uint8_t smem_raw[];
    WideSmem& S = *reinterpret_cast<WideSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int HT = p.H * p.T;
    // Programmatic dependent of the previous kernel on the stream: nothing is
    // read before this point.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    // G = p.row_ctas CTAs per (partition, request), adjacent in the grid, CTA r
    // taking rows [r * p.rows_per_cta, ...): they run at the same time, so all
    // but the first read each page from L2.  In request order the grid's x is
    // (partition, r) and y the request; with more CTAs than SMs the G CTAs of
    // launch entry e take unit e of the longest-first order (lpt_order_kernel).
    const int G = p.row_ctas;
    int crank, split, b, L_known = -1;
    if constexpr (kLpt) {
        const long long k = (long long)blockIdx.y * gridDim.x + blockIdx.x;
        const int2 u = p.lpt_order[k / G];
        if (u.x < 0) return;  // past the last unit with history: nothing to do
        crank = static_cast<int>(k % G);
        b = u.x / p.n_splits;
        split = u.x % p.n_splits;
        L_known = u.y;
    } else {
        crank = static_cast<int>(blockIdx.x % G);
        split = blockIdx.x / G;
        b = blockIdx.y;
    }
    const int r0 = p.rows_per_cta * crank;
    const int HTc = min(p.rows_per_cta, HT - r0);  // rows of this CTA (<= 32)
    volatile int* abort = &S.abort;

    // Loads that depend only on the launch indices go out first: the
    // producer's first 64 page ids, and the query rows of warps 1..19.
    constexpr int kStageWarps = kWThreads / 32 - 1;                   // 19
    constexpr int kQR = (kWRows + kStageWarps - 1) / kStageWarps;     // 2 rows per staging warp
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
            const int r = warp - 1 + kStageWarps * rr;
            const uint4* src = reinterpret_cast<const uint4*>(p.q + ((int64_t)b * HT + r0 + r) * kDqk);
#pragma unroll
            for (int k = 0; k < 3; ++k) {
                const int c = lane + 32 * k;  // 16-byte chunk: 8 bf16 values
                qv[rr][k] = (r < HTc && c < kDqk / 8) ? __ldg(src + c) : make_uint4(0, 0, 0, 0);
            }
        }
    }
    int L = L_known >= 0 ? L_known : __ldg(p.seq_lens + b);
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
        for (int s = 0; s < kWStages; ++s) {
            mbar_init(&S.full[s], 1);
            mbar_init(&S.empty[s], 1);
        }
        for (int i = 0; i < kWSBufs; ++i) {
            mbar_init(&S.s_full[i], 2);              // both K-halves of QK^T
            mbar_init(&S.s_empty[i], 4 * kWGroups);  // every attention warp reads every score tile
        }
        for (int i = 0; i < kWPBufs; ++i) {
            mbar_init(&S.p_full[i], 4 * kWGroups);   // every attention warp writes its rows of P
            mbar_init(&S.pv_done[i], 1);
        }
        for (int i = 0; i < 3; ++i) mbar_init(&S.mma_done[i], 1);
        S.abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    __syncthreads();
    // Page i into slot i % kWStages (one thread); the first pages as nine boxes
    // (first bytes in sooner), later ones as one 3-D copy.
    int issued = 0;
    auto issue_page = [&](int i, int32_t pid) {
        const int s = i % kWStages;
        if (pid < 0 || pid >= p.num_pages) {
            if (crank == 0) atomicCAS(p.err, 0, kErrPageRange);
            pid = 0;  // load a valid page; the attention warps mask and zero it
        }
        mbar_expect_tx(&S.full[s], kWSlotBytes);
        const uint32_t dst = smem_u32(S.slot[s]);
        if (i < kWStages) {
#pragma unroll
            for (int j = 0; j < kWBoxes; ++j)
                tma_load_box(dst + j * kWBoxBytes, &tmap_box, 64 * j, pid * kPage, &S.full[s]);
        } else {
            tma_load_page(dst, &tmap, pid * kPage, &S.full[s]);
        }
    };
    if (warp == 0 && !p.test_stall_copies) {
        const int first = min(kWStages, n_pages);
        for (int i = 0; i < first; ++i) {
            const int32_t pid = __shfl_sync(0xffffffffu, pid_cur, i);
            if (lane == 0) issue_page(i, pid);
        }
        issued = first;
        __syncwarp();
    }
    if (warp == 2) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(&S.tmem_base)),
                     "r"(kWTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    // Query rows r = warp - 1 + 19 k (< 32): exact split q * 2^e = q1 + q2 / 16.
    if (warp > 0) {
#pragma unroll
        for (int rr = 0; rr < kQR; ++rr) {
            const int r = warp - 1 + kStageWarps * rr;
            if (r >= kWRows) continue;
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
                    *reinterpret_cast<uint2*>(S.qp + kmajor_off(kWRows + r, k0, kDqk)) = make_uint2(q2[0], q2[1]);
                }
                if (lane == 0) {
                    S.row_scale[r] = kv_scale * p.sm_scale_log2 * ldexpf(1.f, -e);
                    S.rowlim[r] = (L == 0) ? 0 : L - p.T + 1 + (r0 + r) / p.H;
                }
            } else {
                for (int c = lane; c < kDqk / 8; c += 32) {
                    *reinterpret_cast<uint2*>(S.qp + kmajor_off(r, 8 * c, kDqk)) = make_uint2(0, 0);
                    *reinterpret_cast<uint2*>(S.qp + kmajor_off(kWRows + r, 8 * c, kDqk)) = make_uint2(0, 0);
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
    if (warp > 0) asm volatile("bar.sync %0, %1;" ::"n"(kWSetupBar), "n"(kWThreads - 32) : "memory");
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
                if (!warp_wait(&S.empty[i % kWStages], ((i / kWStages) & 1) ^ 1, abort, p.err)) break;
                if (lane == 0) issue_page(i, pid);
                __syncwarp();
                issued = i + 1;
            }
        }
        if (lane == 0) {
            // never leave with a copy in flight into this CTA's shared memory
            const uint64_t t0 = global_ns();
            for (int i = max(0, issued - kWStages); i < issued; ++i) {
                const int s = i % kWStages;
                const uint32_t par = (i / kWStages) & 1;
                while (!mbar_try_wait(&S.full[s], par) && global_ns() - t0 < kTimeoutNs) {
                }
            }
        }
    } else if (warp == 1 || warp == 3) {
        // ======================= QK^T issuers =======================
        // Both warps take every page: warp 1 the K-steps over dims [0, 288) into
        // the first half of the score tile, warp 3 those over [288, 576) into the
        // second half (one thread needs ~40 cycles per MMA, so the split halves
        // the time to the page's scores).  The whole warp runs the loop, one
        // elected lane issues.  Pages are taken in order, so the parity of a
        // slot's full barrier is exact.
        const int me = warp == 1 ? 0 : 1;
        const bool leader = elect_one();
        const uint64_t qd = smem_desc(smem_u32(S.qp), 128, (kDqk / 16) * 128, kLayoutNone);
        constexpr uint32_t kIdesc = idesc_e4m3(64, kWN, false, false);
        constexpr int kHalf = kDqk / 64;  // 9 K-steps of 32 dims per issuer
        for (int i = 0; i < n_pages; ++i) {
            const int s = i % kWStages, sb = i % kWSBufs;
            if (!warp_wait(&S.full[s], (i / kWStages) & 1, abort, p.err)) break;
            if (!warp_wait(&S.s_empty[sb], ((i / kWSBufs) & 1) ^ 1, abort, p.err)) break;
            tc_fence_after();
            const uint64_t ad = smem_desc(smem_u32(S.slot[s]), 16, 512, kLayoutSw64);
            const uint32_t d = tmem + kWSCols * sb + kWN * me;
            if (leader) {
#pragma unroll
                for (int j = 0; j < kHalf; ++j) {
                    const int ks = kHalf * me + j;
                    mma_e4m3(d, ad + static_cast<uint64_t>(((ks >> 1) * kWBoxBytes + (ks & 1) * 32) >> 4),
                             qd + static_cast<uint64_t>(ks * 16), kIdesc, j > 0);
                }
                mma_commit(&S.s_full[sb]);
            }
            __syncwarp();
        }
        if (leader) {
            mma_commit(&S.mma_done[me]);
            const uint64_t t0 = global_ns();
            while (!mbar_try_wait(&S.mma_done[me], 0) && global_ns() - t0 < kTimeoutNs) {
            }
        }
        __syncwarp();
    } else if (warp == 2) {
        // ======================= PV issuer =======================
        // O[128c + dim][n] += sum_k V^T[dim][k] P[k][n], n < 32 the p1 codes of the
        // rows, n >= 32 their p2 codes; 2 K-steps x 4 dim blocks per page.
        const bool leader = elect_one();
        constexpr uint32_t kIdesc = idesc_e4m3(128, kWN, true, true);
        for (int i = 0; i < n_pages; ++i) {
            const int s = i % kWStages, kb = i % kWPBufs;
            if (!warp_wait(&S.p_full[kb], (i / kWPBufs) & 1, abort, p.err)) break;
            tc_fence_after();
            const uint64_t ad = smem_desc(smem_u32(S.slot[s]), kWBoxBytes, 512, kLayoutSw64);
            // MN-major, no swizzle: LBO = stride between 8-position groups (K),
            // SBO = stride between 16-column core matrices (N).
            const uint64_t bd = smem_desc(smem_u32(S.pp[kb]), kWPpKStride, 128, kLayoutNone);
            if (leader) {
#pragma unroll
                for (int ks = 0; ks < kPage / 32; ++ks)
#pragma unroll
                    for (int c = 0; c < kDv / 128; ++c)
                        mma_e4m3(tmem + kWOCol0 + kWN * c,
                                 ad + static_cast<uint64_t>((2 * c * kWBoxBytes + ks * 32 * 64) >> 4),
                                 bd + static_cast<uint64_t>((ks * 4 * kWPpKStride) >> 4), kIdesc,
                                 i > 0 || ks > 0);
                mma_commit(&S.pv_done[kb]);
                mma_commit(&S.empty[s]);
            }
            __syncwarp();
        }
        if (leader) {
            mma_commit(&S.mma_done[2]);
            const uint64_t t0 = global_ns();
            while (!mbar_try_wait(&S.mma_done[2], 0) && global_ns() - t0 < kTimeoutNs) {
            }
        }
        __syncwarp();
    } else if (warp >= 4) {
        // ======================= attention warpgroups =======================
        // Warpgroup g owns rows [8g, 8g + 8).  In the M = 64 score tile a warp's
        // lanes 0..15 hold its 16 positions; lane l < 16 keeps rows 8g..8g+3 of
        // position l and sends rows 8g+4..8g+7 to lane l + 16, so every lane works
        // on 4 rows of one position.  A row's probabilities are P = 2^(s - r)
        // against a reference r that moves only when a score would exceed
        // r + kWHeadroom; the accumulated output columns of the moved rows are
        // then rescaled in place in TMEM.
        const int g = (warp - 4) >> 2;
        const int quad = warp & 3;
        const int half = lane >> 4;
        const int pr = 16 * quad + (lane & 15);   // position within the page
        const int d = 32 * quad + lane;           // latent dim within each 128-dim block
        const int grow0 = kWRg * g + kWRL * half; // this lane's first row
        const float NEG = -INFINITY;
        const bool causal = p.T > 1;              // for T = 1 the partition end bounds every row
        const uint32_t lane_base = static_cast<uint32_t>(32 * quad) << 16;
        const uint32_t to = tmem + lane_base + kWOCol0 + kWRg * g;  // p1 columns of this group, block 0
        const int32_t* bt = p.block_table + (int64_t)b * p.bt_stride + pg_begin;
        float lp[kWRL], rsc[kWRL], rr[kWRL];
        int lim[kWRL];
        float r_l = NEG;                          // lane h < 8: reference of group row h
#pragma unroll
        for (int j = 0; j < kWRL; ++j) {
            lp[j] = 0.f;
            rr[j] = NEG;
            rsc[j] = S.row_scale[grow0 + j];
            // padding rows (>= HTc) see nothing; T = 1 rows are bounded by the partition
            lim[j] = grow0 + j >= HTc ? -1 : (causal ? S.rowlim[grow0 + j] : INT_MAX);
        }
        bool fail = false;
        int32_t pid_next = __ldg(bt);
        const float ref_shift = p.ref_shift;
        for (int i = 0; i < n_pages; ++i) {
            const int sb = i % kWSBufs, kb = i % kWPBufs, par = i & 1;
            const int32_t pid = pid_next;
            if (i + 1 < n_pages) pid_next = __ldg(bt + i + 1);
            const bool page_ok = pid >= 0 && pid < p.num_pages;
            const int pos = (pg_begin + i) * kPage + pr;
            const bool in_part = page_ok && pos < p_end;
            float s[kWRL];
            bool over = false;  // a score of this lane exceeds its row's reference + headroom
            bool rescale = false;  // a reference moved after the partition's first page
            float a_mv = 1.f;      // lane h < 8: factor for group row h's accumulated columns
#pragma unroll
            for (int j = 0; j < kWRL; ++j) s[j] = NEG;
            // ---- scores of this page ----
            if (!fail) fail = !warp_wait(&S.s_full[sb], (i / kWSBufs) & 1, abort, p.err);
            if (!fail) {
                tc_fence_after();
                uint32_t r1[8], r2[8], r1b[8], r2b[8];
                const uint32_t ta = tmem + lane_base + kWSCols * sb + kWRg * g;
                tmem_ld8(ta, r1);                   // q1 . x over dims [0, 288) of the group's rows
                tmem_ld8(ta + kWRows, r2);          // q2 . x
                tmem_ld8(ta + kWN, r1b);            // the same over dims [288, 576)
                tmem_ld8(ta + kWN + kWRows, r2b);
                tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    r1[j] = __float_as_uint(__uint_as_float(r1[j]) + __uint_as_float(r1b[j]));
                    r2[j] = __float_as_uint(__uint_as_float(r2[j]) + __uint_as_float(r2b[j]));
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&S.s_empty[sb]);
#pragma unroll
                for (int j = 0; j < kWRL; ++j) {
                    const float lo = __uint_as_float(r1[j]) + __uint_as_float(r2[j]) * 0.0625f;
                    const float hi = __uint_as_float(r1[kWRL + j]) + __uint_as_float(r2[kWRL + j]) * 0.0625f;
                    const float moved = __shfl_xor_sync(0xffffffffu, hi, 16);
                    const float v = (half ? moved : lo) * rsc[j];
                    s[j] = (in_part && pos < lim[j]) ? v : NEG;
                    over |= s[j] > rr[j] + kWHeadroom;  // rr = -inf: any score moves it
                }
            }
            // One barrier per page decides whether any row's reference moves; only
            // then are the page maxima reduced (a second barrier).
            if (group_sync_or(g, fail || over)) {
                if (!fail) {
                    float mine = NEG;  // lane 16 half + j (j < 4): this warp's max of row 4 half + j
#pragma unroll
                    for (int j = 0; j < kWRL; ++j) {
                        const float wlo = warp_max_redux(half ? NEG : s[j]);
                        const float whi = warp_max_redux(half ? s[j] : NEG);
                        mine = ((lane & 15) == j) ? (half ? whi : wlo) : mine;
                    }
                    if ((lane & 15) < kWRL) S.red_m[g][par][kWRL * half + (lane & 15)][quad] = mine;
                }
                if (group_sync_or(g, fail)) {
                    fail = true;
                    break;
                }
                float t = NEG;
                if (lane < kWRg) {
                    const float4 vm = *reinterpret_cast<const float4*>(S.red_m[g][par][lane]);
                    t = fmaxf(fmaxf(vm.x, vm.y), fmaxf(vm.z, vm.w));
                }
                const bool need = lane < kWRg && t > r_l + kWHeadroom;
                if (__ballot_sync(0xffffffffu, need)) {
                    const float rn = need ? t - ref_shift : r_l;
                    const float a = need ? exp2f(r_l - rn) : 1.f;  // r_l = -inf: nothing to keep
                    r_l = rn;
                    if (p.test_counts && quad == 0 && lane == 0) {
                        atomicAdd(p.test_counts + 1, 1);
                        if (i > 0) atomicAdd(p.test_counts, 1);
                    }
#pragma unroll
                    for (int j = 0; j < kWRL; ++j) {
                        rr[j] = __shfl_sync(0xffffffffu, rn, kWRL * half + j);
                        lp[j] *= __shfl_sync(0xffffffffu, a, kWRL * half + j);
                    }
                    if (i > 0) {  // the accumulated columns are rescaled below
                        rescale = true;
                        a_mv = a;
                    }
                }
            }
            // ---- probabilities of this page -> this group's rows of [p1 | p2] ----
            if constexpr (kWPBufs < kWStages) {
                if (!fail && i >= kWPBufs)
                    fail = !warp_wait(&S.pv_done[kb], ((i / kWPBufs) - 1) & 1, abort, p.err);
            }
            if (!fail) {
#pragma unroll
                for (int j = 0; j < kWRL; ++j) {
                    s[j] = (s[j] == NEG) ? 0.f : fast_exp2(s[j] - rr[j]);
                    lp[j] += s[j];
                }
                uint32_t c1a, c2a, c1b, c2b;
                wsplit_p(s[0], s[1], c1a, c2a);
                wsplit_p(s[2], s[3], c1b, c2b);
                uint8_t* pp = S.pp[kb];
                *reinterpret_cast<uint32_t*>(pp + wpp_off(grow0, pr)) = (c1a & 0xffffu) | (c1b << 16);
                *reinterpret_cast<uint32_t*>(pp + wpp_off(kWRows + grow0, pr)) = (c2a & 0xffffu) | (c2b << 16);
                // Positions past the partition's end (or of a page whose id was out
                // of range) may hold anything, even NaN codes: zero them so that
                // 0 * x stays 0 in the PV product.  Their QK^T is already done.
                if (g == 0 && half == 0 && !in_part) {
                    uint8_t* row = S.slot[i % kWStages] + pr * 64;
#pragma unroll
                    for (int j = 0; j < kWBoxes; ++j) {
                        uint4* q4 = reinterpret_cast<uint4*>(row + j * kWBoxBytes);
                        q4[0] = q4[1] = q4[2] = q4[3] = make_uint4(0, 0, 0, 0);
                    }
                }
                if (rescale) {
                    // The tile holds PV of pages 0..i-1: wait for the last one (the
                    // probabilities above overlapped that wait), then scale this
                    // group's p1 and p2 columns (every warp its lane quadrant).
                    const int pk = (i - 1) % kWPBufs;
                    if (!warp_wait(&S.pv_done[pk], ((i - 1) / kWPBufs) & 1, abort, p.err)) {
                        fail = true;
                    } else {
                        tc_fence_after();
                        float al[kWRg];
#pragma unroll
                        for (int j = 0; j < kWRg; ++j) al[j] = __shfl_sync(0xffffffffu, a_mv, j);
#pragma unroll
                        for (int c = 0; c < 4; ++c) {
#pragma unroll
                            for (int u = 0; u < 2; ++u) {
                                uint32_t v[8];
                                tmem_ld8(to + kWN * c + kWRows * u, v);
                                tmem_wait_ld();
#pragma unroll
                                for (int j = 0; j < kWRg; ++j)
                                    v[j] = __float_as_uint(__uint_as_float(v[j]) * al[j]);
                                tmem_st8(to + kWN * c + kWRows * u, v);
                            }
                        }
                        tmem_wait_st();
                    }
                }
                if (!fail) {
                    fence_async_smem();
                    tc_fence_before();  // TMEM stores of a rescale precede the next PV
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&S.p_full[kb]);
                }
            }
        }

        // ---- this group's rows: normaliser, log-sum-exp, output ----
        bool o_ok = !fail;
        if (o_ok)
            o_ok = warp_wait(&S.pv_done[(n_pages - 1) % kWPBufs], ((n_pages - 1) / kWPBufs) & 1, abort, p.err);
        {
            float e[kWRg];
#pragma unroll
            for (int h = 0; h < kWRg; ++h) e[h] = ((h >> 2) == half) ? lp[h & 3] : 0.f;
            const float wsum = warp_transpose_sum8(e, lane);
            if ((lane & 3) == 0) S.red_l[g][lane >> 2][quad] = wsum;
        }
        const bool bad = group_sync_or(g, !o_ok);  // partials written; failure anywhere in the group
        float w = 0.f;                            // lane h < 8: weight of group row h
        if (lane < kWRg) {
            const float4 vl = *reinterpret_cast<const float4*>(S.red_l[g][lane]);
            const float l = (vl.x + vl.y) + (vl.z + vl.w);
            w = (l > 0.f && !bad) ? kv_scale / l : 0.f;
            const int row = kWRg * g + lane;
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
        float wj[kWRg];
#pragma unroll
        for (int j = 0; j < kWRg; ++j) wj[j] = __shfl_sync(0xffffffffu, w, j);
        if (!bad) tc_fence_after();
        const int64_t row0 = (int64_t)b * HT + r0;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            uint32_t v1[8], v2[8];
            if (!bad) {
                tmem_ld8(to + kWN * c, v1);
                tmem_ld8(to + kWN * c + kWRows, v2);
                tmem_wait_ld();
            } else {
#pragma unroll
                for (int j = 0; j < kWRg; ++j) v1[j] = v2[j] = 0u;
            }
#pragma unroll
            for (int j = 0; j < kWRg; ++j) {
                const int row = kWRg * g + j;
                if (row < HTc) {
                    const float o = fmaf(__uint_as_float(v2[j]), 0.0625f, __uint_as_float(v1[j])) * wj[j];
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
    if (warp == 2) {
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(S.tmem_base), "r"(kWTmemCols)
                     : "memory");
    }
}
}  // namespace

// ---------------------------------------------------------------- host side

// Launch the wide kernel: p.row_ctas CTAs per (partition, request), each of at
// most 32 rows (p.rows_per_cta); the maps are those of the 12-head kernel
// (3-D page view and 2-D box view of the cache).
cudaError_t launch_tc_wide(const DecodeParams& p, const CUtensorMap& map, const CUtensorMap& map_box, bool lpt,
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
            if ((e = cudaFuncSetAttribute(tc_wide_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          (int)sizeof(WideSmem) + 1024)) != cudaSuccess ||
                (e = cudaFuncSetAttribute(tc_wide_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          (int)sizeof(WideSmem) + 1024)) != cudaSuccess)
                return e;
            ready[dev] = true;
        }
    }
    if (p.rows_per_cta < 1 || p.rows_per_cta > kWRows || p.row_ctas < 1 ||
        (int64_t)p.rows_per_cta * p.row_ctas < (int64_t)p.H * p.T)
        return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(p.row_ctas) * static_cast<unsigned>(p.n_splits),
                       static_cast<unsigned>(p.B));
    cfg.blockDim = dim3(kWThreads);
    cfg.dynamicSmemBytes = sizeof(WideSmem) + 1024;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = lpt ? cudaLaunchKernelEx(&cfg, tc_wide_kernel<true>, map, map_box, p)
            : cudaLaunchKernelEx(&cfg, tc_wide_kernel<false>, map, map_box, p);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace mla
