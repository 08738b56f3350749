// mla_tc.cu -- tcgen05 tensor-core split-KV MLA decode over a paged FP8 latent
// cache, for sm_103a (GB300): the kernel for units of up to 16 query rows
// (H * T <= 16, e.g. 12 heads x 1 position), and the dispatch to the wide
// kernel (mla_tc_wide.cu) for 17..128 rows.
//
// Method: "Kimi K3 on AMD Instinct MI355X" post -- section 4 (the history is
// cut into parallel partitions inside one GPU and the partial results are
// combined; KV storage is unchanged), section 1 (each partial answer carries
// its log-sum-exp so partials merge exactly), benchmark section (FP8 KV).
//
// Design (GB300-first):
//   * The FP8 codes are MMA operands as they sit in the cache: every 64-position
//     page is bulk-copied by TMA (one 3-D box, or for the first pages nine 2-D
//     boxes, landing as nine 64x64-byte tiles with 64-byte swizzle) into a
//     5-deep shared-memory ring and consumed by tcgen05.mma kind::f8f6f4 with no
//     dequantisation pass.  kv_scale is folded into the score scale and the
//     output scale.
//   * The bf16 query is split exactly into two e4m3 terms per row,
//     q * 2^e = q1 + q2 / 16, with a per-row power of two e that maps max|q| to
//     (224, 448]; the 576-dim dot products are S1 = q1.x and S2 = q2.x as two
//     column blocks of one MMA.
//   * Swap-AB: positions are the MMA M dimension.  QK^T: D[64 pos x 32] =
//     K_page[64 x 576] . [q1 | q2]^T (M=64, N=32).  PV: for each 128-dim block of
//     the latent, D[128 dims x 32] = V^T[128 x 64 pos] . [p1 | p2]^T, with V^T read
//     from the same page tile as an MN-major operand (M=128, N=32).
//   * Probabilities are taken against a per-head reference r that moves only
//     when a score would exceed r + 8.8 (log2 units): P = 2^(s - r) in (0, 445],
//     stored as two e4m3 terms p1 + p2 / 16 (relative error ~2^-8, the bf16
//     level).  Each lane first compares its own scores with r; one named
//     barrier ORs that test over the warpgroup, and only when it is set do the
//     warps reduce the page maxima and move r (new r = page max - S), rescaling
//     the accumulated output in TMEM in place.  Most pages skip the reductions.
//     The shift S (4..7, p.ref_shift) bounds what e4m3's subnormal floor can
//     take: each p1 + p2/16 is off by at most ~2^-14 in absolute terms, i.e.
//     2^-(14+S) of the row's largest weight, so the n positions a warpgroup
//     accumulates lose at most n * 2^-(14+S) of it together; the host picks
//     S = log2(n) - 6 within [4, 7] (at most 2^-8 lost), since every further
//     unit of S makes references move more often.  The rescale of a move waits
//     for the previous PV, so it runs after the page's probabilities are
//     written, overlapping that wait.
//   * Warp roles: warp 0 TMA producer; three MMA-issuing warps (warp 1: QK^T of
//     even pages, warp 3: QK^T of odd pages, warp 2: PV of every page), because
//     one thread can issue a tcgen05.mma only every ~50 cycles; and two
//     attention warpgroups (warps 4-7, 8-11) that take alternate pages.  For
//     its page a warpgroup reads the score tile (TMEM lane = position), forms
//     the probabilities and hands them to the PV issuer; PV accumulates into
//     that warpgroup's own output tile in TMEM (lane = latent dim) over all of
//     its pages.  Each thread keeps fp32 partial normalisers of its positions.
//   * At the end the warpgroup without the last page hands over its references
//     and normalisers; the other reads both tiles from TMEM, combines them and
//     stores the rows.
//   * Every wait is bounded; on timeout the kernel records an error, drains its
//     own copies and MMAs, frees TMEM and returns.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include <cmath>
#include <mutex>

#include "mla_internal.cuh"
#include "mla_tc_ptx.cuh"

namespace mla {
namespace {

constexpr int kGroups = 2;                   // attention warpgroups
constexpr int kThreads = 128 + 128 * kGroups;
constexpr int kStages = 5;                   // page slots in the TMA ring
constexpr int kNq = 16;                      // rows (t, h) per CTA, padded
constexpr int kNqk = 2 * kNq;                // MMA N: q1 rows | q2 rows (and p1 | p2)
constexpr int kMaxRowsTc = 128;             // rows beyond 16 go to the wide kernel
constexpr int kWideRows = 32;               // rows per CTA of the wide kernel (at most 64)
constexpr int kSlotBytes = kPage * kDqk;     // 36,864: one page
constexpr int kBoxBytes = kPage * 64;        // 4,096: 64 positions x 64 dims
constexpr int kBoxes = kDqk / 64;            // 9
constexpr int kQpBytes = kNqk * kDqk;        // 18,432
constexpr int kPpBytes = kNqk * kPage;       // 2,048
constexpr int kSBufs = 4;                    // score tiles in TMEM (QK^T look-ahead)
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kSCol0 = 0;               // S buffers: 4 x 32 cols at [0, 128)
constexpr uint32_t kSCols = 32;
constexpr uint32_t kOCol0 = 128;             // O buffers: one per warpgroup, 128 cols each
constexpr int kLptMaxB = 1024;               // longest-first launches order at most this many requests
constexpr int kLptThreads = 1024;            // the ordering kernel: one thread per request
// log2 units a score may exceed its head's reference: P = 2^(s - r) <= 2^8.8 < 448
constexpr float kHeadroom = 8.8f;
static_assert(kOCol0 + 128 * kGroups <= kTmemCols, "TMEM budget");


struct Smem {
    uint8_t slot[kStages][kSlotBytes];       // 1024-aligned page tiles
    uint8_t qp[kQpBytes];                    // [q1 | q2] K-major, no swizzle
    uint8_t pp[kGroups][2][kPpBytes];        // [p1 | p2] MN-major, no swizzle, per group page
    float red_m[kGroups][2][kNq][4];         // [group][iter parity][head][warp] tile maxima
    float red_l[kGroups][kNq][4];            // per group: end-of-loop normaliser partials
    float fin[2][kNq];                       // other warpgroup: final reference / normaliser by head
    int fin_bad;                             // the other warpgroup's tile is incomplete (a wait gave up)
    alignas(16) float row_scale[kNq];        // kv_scale * sm_scale * log2(e) * 2^-e
    alignas(16) int rowlim[kNq];             // visible prefix per row; -1 = padding
    uint64_t full[kStages], empty[kStages];
    uint64_t s_full[kSBufs], s_empty[kSBufs];
    uint64_t p_full[kGroups][2];             // group's probabilities of its page are ready
    uint64_t pv_done[kGroups][2];            // group's PV of its page k done (buffer k & 1)
    uint64_t fin_l_bar[kGroups];             // group's normaliser partials are written
    uint64_t mma_done[3];                    // per MMA-issuing thread: its MMAs drained
    uint32_t tmem_base;
    int abort;
};
static_assert(sizeof(uint8_t[kStages][kSlotBytes]) % 1024 == 0, "slots keep 1 KB alignment");

constexpr uint32_t kIdescQK = idesc_e4m3(64, kNqk, false, false);
constexpr uint32_t kIdescPV = idesc_e4m3(128, kNqk, true, true);

// Byte offset of (column n, position k) in the probability operand [p1 | p2]:
// MN-major, no swizzle.  A core matrix is 8 positions x 16 columns (one
// 16-byte row per position); the p1 and p2 core matrices of an 8-position
// group sit side by side (128 B apart), and groups follow every 256 B.  One
// position's 16 p1 codes are thus one 16-byte store, and so are its p2 codes.
constexpr uint32_t kPpMnStride = 128;  // between the p1 and p2 core matrices
constexpr uint32_t kPpKStride = 256;   // between 8-position groups
__device__ __forceinline__ uint32_t pp_off(int n, int k) {
    return (n >> 4) * kPpMnStride + (n & 15) + (k & 7) * 16 + (k >> 3) * kPpKStride;
}

// Two probabilities (times 256) -> e4m3 codes of p1 and of 16 * (value - p1),
// computed in f16 (11 significant bits cover the 8 that p1 + p2/16 keeps).
__device__ __forceinline__ void split_p(float a0, float a1, uint32_t& c1, uint32_t& c2) {
    const __half2 h = __floats2half2_rn(a0, a1);
    const __half2_raw hr = *reinterpret_cast<const __half2_raw*>(&h);
    c1 = static_cast<uint32_t>(__nv_cvt_halfraw2_to_fp8x2(hr, __NV_SATFINITE, __NV_E4M3));
    const __half2_raw br = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(c1), __NV_E4M3);
    const __half2 back = *reinterpret_cast<const __half2*>(&br);
    const __half2 r = __hmul2(__hsub2(h, back), __float2half2_rn(16.f));
    c2 = static_cast<uint32_t>(
        __nv_cvt_halfraw2_to_fp8x2(*reinterpret_cast<const __half2_raw*>(&r), __NV_SATFINITE, __NV_E4M3));
}

// Longest-first launches (more units than SMs): the order of all B * n_splits
// (request, partition) units, computed once per call by one CTA from the
// device-resident lengths, before the decode kernel (which waits for it).
// Full-chunk units come first (request-major), then each request's partial
// chunk, longest remainder first (ties: lower request first); the decode CTAs
// are dispatched in launch order, so the SMs that free up take the longest
// units left and end within about one short unit of each other.  Entry k is
// {b * n_splits + split, seq_len of b}, or {-1, 0} past the last unit with
// history.  Nothing is written for the empty units (partitions past a
// request's end): the split combine counts the partitions past a request's
// history as empty.  A length outside [0, 64 * max_pages], or in (0, T),
// reads nothing and sets device error 3.
__global__ void __launch_bounds__(kLptThreads, 1) lpt_order_kernel(const DecodeParams p) {
    __shared__ int full_pfx[kLptMaxB + 1];
    __shared__ int rem_s[kLptMaxB];
    __shared__ int warp_sum[kLptThreads / 32];
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;");  // they wait for this grid to finish
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int B = p.B, chunk = p.chunk_pages, n_splits = p.n_splits;
    int L = 0, full = 0, rem = 0;
    if (tid < B) {
        L = __ldg(p.seq_lens + tid);
        if (L < 0 || L > p.max_pages * kPage || (L > 0 && L < p.T)) {
            atomicCAS(p.err, 0, kErrSeqRange);
            L = 0;
        }
        const int pages = (L + kPage - 1) / kPage;
        full = pages / chunk;
        rem = pages - full * chunk;
        rem_s[tid] = rem;
    }
    // exclusive prefix over the requests of their full-chunk units
    int x = full;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, d);
        if (lane >= d) x += y;
    }
    if (lane == 31) warp_sum[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int w = warp_sum[lane];
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, w, d);
            if (lane >= d) w += y;
        }
        warp_sum[lane] = w;  // inclusive prefix of the warps' sums
    }
    __syncthreads();
    x += warp > 0 ? warp_sum[warp - 1] : 0;  // inclusive prefix of this request
    if (tid < B) full_pfx[tid] = x - full;
    if (tid == kLptThreads - 1) full_pfx[B] = x;  // every full unit (threads >= B add 0)
    const int n_part = __syncthreads_count(tid < B && rem > 0);  // also publishes full_pfx and rem_s
    const int n_full = full_pfx[B];
    int2* order = p.lpt_order;
    if (tid < B) {
        for (int sp = 0; sp < full; ++sp) order[full_pfx[tid] + sp] = make_int2(tid * n_splits + sp, L);
        if (rem > 0) {
            int ahead = 0;  // partial chunks ordered before this one
            for (int o = 0; o < B; ++o) {
                const int r2 = rem_s[o];
                ahead += (r2 > rem || (r2 == rem && o < tid)) ? 1 : 0;
            }
            order[n_full + ahead] = make_int2(tid * n_splits + full, L);
        }
    }
    for (int k = n_full + n_part + tid; k < B * n_splits; k += kLptThreads) order[k] = make_int2(-1, 0);
}

// One (request b, partition split) unit, start to finish: barriers, TMEM,
// query operand, the warp roles, the epilogue, and a last barrier after which
// every copy and MMA has drained.  Returns false (having written an empty
// partial and allocated nothing) when the unit holds no history.
template <int kRows>
__device__ __forceinline__ bool decode_unit(const CUtensorMap* tmap, const CUtensorMap* tmap_box,
                                            const DecodeParams& p, Smem& S, int b, int split, int L_known) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int HT = p.H * p.T;
    const int HTc = HT;                          // rows of every unit (all of the request's)
    volatile int* abort = &S.abort;
    // Global loads that depend only on the launch indices go out together,
    // before any of their values is needed: the producer's first 64 page ids
    // (one per lane, in two windows of 32) and the query rows of warps 1..11.
    const int pg_begin = split * p.chunk_pages;
    const int32_t* bt_cta = p.block_table + (int64_t)b * p.bt_stride + pg_begin;
    int32_t pid_cur = 0, pid_nxt = 0;
    uint4 qv[2][3];  // rows warp - 1 and warp + 10, 16-byte chunks lane + 32k
    if (warp == 0) {
        if (lane == 0) {
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tmap_box)) : "memory");
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tmap)) : "memory");
        }
        pid_cur = pg_begin + lane < p.max_pages ? __ldg(bt_cta + lane) : 0;
        pid_nxt = pg_begin + 32 + lane < p.max_pages ? __ldg(bt_cta + 32 + lane) : 0;
    } else {
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
            const int r = warp - 1 + (kThreads / 32 - 1) * rr;
            const uint4* src = reinterpret_cast<const uint4*>(p.q + ((int64_t)b * HT + r) * kDqk);
#pragma unroll
            for (int k = 0; k < 3; ++k) {
                const int c = lane + 32 * k;  // 16-byte chunk: 8 bf16 values
                qv[rr][k] = (r < kNq && r < HTc && c < kDqk / 8) ? __ldg(src + c) : make_uint4(0, 0, 0, 0);
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
        // None of this request's history falls in this partition: leave before
        // any set-up.  Its rows get lse = -inf, a partial the merge skips, or,
        // unsplit, out = 0 and lse = -inf.
        const int64_t row0 = (int64_t)b * HT;
        if (p.n_splits == 1) {
            for (int idx = tid; idx < HTc * kDv; idx += kThreads) p.out[row0 * kDv + idx] = 0;
            if (p.lse)
                for (int idx = tid; idx < HTc; idx += kThreads) p.lse[row0 + idx] = -INFINITY;
        } else {
            for (int idx = tid; idx < HTc; idx += kThreads)
                p.part_lse[(int64_t)split * p.B * HT + row0 + idx] = -INFINITY;
        }
        return false;
    }

    // ---------------- set-up: barriers, TMEM, query operand ----------------
    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&S.full[s], 1);
            mbar_init(&S.empty[s], 1);
        }
        for (int i = 0; i < kSBufs; ++i) {
            mbar_init(&S.s_full[i], 1);
            mbar_init(&S.s_empty[i], 4);
        }
        for (int g = 0; g < kGroups; ++g) {
            mbar_init(&S.fin_l_bar[g], 4);
            for (int i = 0; i < 2; ++i) {
                mbar_init(&S.pv_done[g][i], 1);
                mbar_init(&S.p_full[g][i], 4);
            }
        }
        for (int i = 0; i < 3; ++i) mbar_init(&S.mma_done[i], 1);
        S.abort = 0;
        S.fin_bad = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    __syncthreads();  // barriers initialised
    // The producer (warp 0) starts the first copies at once and takes no part in
    // the rest of the set-up: issuing a copy can stall its thread for a long
    // time, and the other warps prepare the query and TMEM meanwhile.
    int issued = 0;
    // Page i into slot i % kStages (one thread).  The first kStages pages go
    // as nine separate boxes, which gets the first bytes in sooner; later pages
    // as one copy instruction, which keeps the producer's issue cost low.
    auto issue_page = [&](int i, int32_t pid) {
        const int s = i % kStages;
        if (pid < 0 || pid >= p.num_pages) {
            atomicCAS(p.err, 0, kErrPageRange);
            pid = 0;  // load a valid page; the softmax masks and zeroes it
        }
        mbar_expect_tx(&S.full[s], kSlotBytes);
        const uint32_t dst = smem_u32(S.slot[s]);
        if (i < kStages) {
#pragma unroll
            for (int j = 0; j < kBoxes; ++j) tma_load_box(dst + j * kBoxBytes, tmap_box, 64 * j, pid * kPage, &S.full[s]);
        } else {
            tma_load_page(dst, tmap, pid * kPage, &S.full[s]);
        }
    };
    if (warp == 0 && n_pages > 0 && !p.test_stall_copies) {
        const int first = min(kStages, n_pages);  // fresh slots: nothing to wait for
        for (int i = 0; i < first; ++i) {
            const int32_t pid = __shfl_sync(0xffffffffu, pid_cur, i);
            if (lane == 0) issue_page(i, pid);
        }
        issued = first;
        __syncwarp();
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(&S.tmem_base)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }

    // Query rows: warps 1..11 prepare rows warp - 1 and warp + 10 (< 16).
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
        const int r = warp - 1 + (kThreads / 32 - 1) * rr;
        if (warp == 0 || r >= kNq) continue;
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
                const int k0 = 8 * c;  // first element of this chunk
                *reinterpret_cast<uint2*>(S.qp + kmajor_off(r, k0, kDqk)) = make_uint2(q1[0], q1[1]);
                *reinterpret_cast<uint2*>(S.qp + kmajor_off(kNq + r, k0, kDqk)) = make_uint2(q2[0], q2[1]);
            }
            if (lane == 0) {
                S.row_scale[r] = kv_scale * p.sm_scale_log2 * ldexpf(1.f, -e);
                S.rowlim[r] = (L == 0) ? 0 : L - p.T + 1 + r / p.H;
            }
        } else {
            for (int c = lane; c < kDqk / 8; c += 32) {
                *reinterpret_cast<uint2*>(S.qp + kmajor_off(r, 8 * c, kDqk)) = make_uint2(0, 0);
                *reinterpret_cast<uint2*>(S.qp + kmajor_off(kNq + r, 8 * c, kDqk)) = make_uint2(0, 0);
            }
            if (lane == 0) {
                S.row_scale[r] = 0.f;
                S.rowlim[r] = -1;
            }
        }
    }
    fence_async_smem();  // query operand: generic writes -> tensor-core reads
    tc_fence_before();
    if (warp > 0) asm volatile("bar.sync 3, %0;" ::"n"(kThreads - 32) : "memory");  // warps 1..11
    tc_fence_after();
    const uint32_t tmem = warp > 0 ? S.tmem_base : 0u;
    asm volatile("griddepcontrol.launch_dependents;");

    if (warp == 0) {
        // ======================= TMA producer =======================
        if (n_pages > 0 && !p.test_stall_copies) {
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
        if (lane == 0 && n_pages > 0) {
            // Drain: never leave with a copy in flight into this CTA's shared memory
            // (one deadline for all of them).
            const uint64_t t0 = global_ns();
            for (int i = max(0, issued - kStages); i < issued; ++i) {
                const int s = i % kStages;
                const uint32_t par = (i / kStages) & 1;
                while (!mbar_try_wait(&S.full[s], par) && global_ns() - t0 < kTimeoutNs) {
                }
            }
        }
    } else if (warp == 1 || warp == 3) {
        // ======================= QK^T issuers =======================
        // Issuing one tcgen05.mma costs the issuing thread tens of cycles, so
        // the MMAs are spread over three threads: warp 1 issues QK^T of the
        // even pages, warp 3 of the odd pages, warp 2 all PV.  Each thread
        // commits only to barriers that it alone signals.
        // The whole warp runs the loop (descriptors stay warp-uniform); one
        // elected lane issues the MMAs and their commit.
        if (n_pages > 0) {
            const bool leader = elect_one();
            const uint64_t qd = smem_desc(smem_u32(S.qp), 128, (kDqk / 16) * 128, kLayoutNone);
            for (int i = (warp == 1 ? 0 : 1); i < n_pages; i += 2) {
                const int sb = i % kSBufs;
                // With an odd ring, slot i % kStages last held page i - kStages of
                // the other issuer.  A parity test of full[] is exact only if that
                // page's phase has completed, so first wait for its PV (which also
                // gates the copy of page i): without it a parity two phases behind
                // would read as complete.
                if (i >= kStages && !warp_wait(&S.empty[i % kStages], ((i / kStages) & 1) ^ 1, abort, p.err))
                    break;
                if (!warp_wait(&S.full[i % kStages], (i / kStages) & 1, abort, p.err)) break;
                if (!warp_wait(&S.s_empty[sb], ((i / kSBufs) & 1) ^ 1, abort, p.err)) break;
                tc_fence_after();
                const uint64_t ad = smem_desc(smem_u32(S.slot[i % kStages]), 16, 512, kLayoutSw64);
                const uint32_t d = tmem + kSCol0 + kSCols * sb;
                if (leader) {
#pragma unroll
                    for (int ks = 0; ks < kDqk / 32; ++ks)
                        mma_e4m3(d, ad + static_cast<uint64_t>(((ks >> 1) * kBoxBytes + (ks & 1) * 32) >> 4),
                                 qd + static_cast<uint64_t>(ks * 16), kIdescQK, ks > 0);
                    mma_commit(&S.s_full[sb]);
                }
                __syncwarp();
            }
            if (leader) {
                mma_commit(&S.mma_done[warp == 1 ? 0 : 1]);
                const uint64_t t0 = global_ns();
                while (!mbar_try_wait(&S.mma_done[warp == 1 ? 0 : 1], 0) && global_ns() - t0 < kTimeoutNs) {
                }
            }
            __syncwarp();
        }
    } else if (warp == 2) {
        // ======================= PV issuer =======================
        // Warpgroup g's output tile accumulates over all of g's pages.
        if (n_pages > 0) {
            const bool leader = elect_one();
            for (int i = 0; i < n_pages; ++i) {
                const int g = i % kGroups, k = i / kGroups, s = i % kStages;
                if (!warp_wait(&S.p_full[g][k & 1], (k >> 1) & 1, abort, p.err)) break;
                tc_fence_after();
                const uint64_t ad = smem_desc(smem_u32(S.slot[s]), kBoxBytes, 512, kLayoutSw64);
                // MN-major, no swizzle: LBO = stride between 8-position groups (K),
                // SBO = stride between the 16-column core matrices (N).
                const uint64_t bd = smem_desc(smem_u32(S.pp[g][k & 1]), kPpKStride, kPpMnStride, kLayoutNone);
                // K-step outer, 128-dim block inner: four independent accumulators.
                if (leader) {
#pragma unroll
                    for (int ks = 0; ks < kPage / 32; ++ks)
#pragma unroll
                        for (int c = 0; c < kDv / 128; ++c)
                            mma_e4m3(tmem + kOCol0 + 128 * g + 32 * c,
                                     ad + static_cast<uint64_t>((2 * c * kBoxBytes + ks * 32 * 64) >> 4),
                                     bd + static_cast<uint64_t>((ks * 4 * kPpKStride) >> 4), kIdescPV,
                                     k > 0 || ks > 0);
                    mma_commit(&S.pv_done[g][k & 1]);
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
        }
    } else if (warp >= 4) {
        // ======================= attention warpgroups =======================
        // Warpgroup g = (warp - 4) / 4 owns pages i = g, g + kGroups, ...  Its
        // output tile accumulates in TMEM over all of those pages against a
        // per-head reference r: the probabilities are P = 2^(s - r), and r moves
        // only when a score would exceed r + kHeadroom, in which case the
        // accumulated tile is rescaled in place.  The four warps of a group meet
        // once per page at a named barrier that also ORs their failure flags, so
        // they always leave the loop together; every other wait is a bounded
        // mbarrier wait.
        const int g = (warp - 4) >> 2;
        const int quad = warp & 3;               // TMEM lane quadrant of this warp
        // The M=64 score tile holds 16 positions per TMEM lane quadrant (lanes
        // 0..15).  Lane l < 16 keeps heads 0..7 of position l, and lane l + 16
        // receives heads 8..15 of the same position: every lane of the warp
        // works on 8 heads of one position.
        const int half = lane >> 4;              // 0: heads 0..7, 1: heads 8..15
        const int pr = 16 * quad + (lane & 15);  // position within the page
        const int d = 32 * quad + lane;          // latent dim within each 128-dim block
        const float NEG = -INFINITY;
        const bool causal = p.T > 1;             // for T = 1 the partition end bounds every row
        const uint32_t to = tmem + (static_cast<uint32_t>(32 * quad) << 16) + kOCol0 + 128 * g;
        const int32_t* bt = p.block_table + (int64_t)b * p.bt_stride + pg_begin;
        // Per lane, for its 8 heads h = 8 * half + j: normaliser partial, score
        // scale and reference (heads >= kRows are padding).
        constexpr int kHL = 8;
        float lp[kHL], rsc[kHL], rr[kHL];
        float r_l = NEG;                         // lane h < kRows: reference of head h
#pragma unroll
        for (int j = 0; j < kHL; ++j) {
            const int h = kHL * half + j;
            lp[j] = 0.f;
            rr[j] = NEG;
            rsc[j] = h < kRows ? S.row_scale[h] : 0.f;
        }
        bool fail = false;
        int k = 0;
        int32_t pid_next = g < n_pages ? __ldg(bt + g) : 0;
        const float ref_shift = p.ref_shift;
        for (int i = g; i < n_pages; i += kGroups, ++k) {
            const int sb = i % kSBufs;           // score buffer
            const int kb = k & 1;                // this group's probability / statistics buffer
            const int32_t pid = pid_next;
            if (i + kGroups < n_pages) pid_next = __ldg(bt + i + kGroups);
            const bool page_ok = pid >= 0 && pid < p.num_pages;
            const int pos = (pg_begin + i) * kPage + pr;
            float s[kHL];
            bool over = false;  // a score of this lane exceeds its head's reference + headroom
            bool rescale = false;  // a reference moved after this group's first page
            float a_mv = 1.f;      // lane h < 16: factor for head h's accumulated columns
            // ---- scores of this page ----
            if (!fail) fail = !warp_wait(&S.s_full[sb], (i / kSBufs) & 1, abort, p.err);
            if (!fail) {
                tc_fence_after();
                uint32_t r1[16], r2[16];
                const uint32_t ta = tmem + (static_cast<uint32_t>(32 * quad) << 16) + kSCol0 + kSCols * sb;
                tmem_ld16(ta, r1);
                tmem_ld16(ta + 16, r2);
                tmem_wait_ld();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&S.s_empty[sb]);
                const bool in_part = page_ok && pos < p_end;
#pragma unroll
                for (int j = 0; j < kHL; ++j) {
                    const int h = kHL * half + j;
                    // S1 + S2/16 of heads j (kept) and 8 + j (sent to lane + 16)
                    const float lo = __uint_as_float(r1[j]) + __uint_as_float(r2[j]) * 0.0625f;
                    const float hi = __uint_as_float(r1[8 + j]) + __uint_as_float(r2[8 + j]) * 0.0625f;
                    const float moved = __shfl_xor_sync(0xffffffffu, hi, 16);
                    const float v = (half ? moved : lo) * rsc[j];
                    s[j] = (h < kRows && in_part && (!causal || pos < S.rowlim[h])) ? v : NEG;
                    over |= s[j] > rr[j] + kHeadroom;  // rr = -inf: any score moves it
                }
            }
            // One barrier per page decides whether any head's reference moves;
            // only then do the warps exchange their page maxima (a second
            // barrier), so most pages skip the max reductions entirely.
            if (group_sync_or(g, fail || over)) {
                if (!fail) {
                    float mine = NEG;  // lanes 8*half + j (j < 8): this warp's max of head 8*half + j
#pragma unroll
                    for (int j = 0; j < kHL; ++j) {
                        // head j of half 0 and head 8 + j of half 1: one full-warp
                        // reduction each, the other half contributing -inf
                        const float wlo = warp_max_redux(half ? NEG : s[j]);
                        const float whi = warp_max_redux(half ? s[j] : NEG);
                        mine = ((lane & 15) == j) ? (half ? whi : wlo) : mine;
                    }
                    if ((lane & 15) < kHL) S.red_m[g][kb][kHL * half + (lane & 15)][quad] = mine;  // rows >= kRows: -inf
                }
                if (group_sync_or(g, fail)) {
                    fail = true;
                    break;
                }
                // ---- page maxima; move the reference where a score would overflow ----
                float t = NEG;
                if (lane < kNq) {
                    const float4 vm = *reinterpret_cast<const float4*>(S.red_m[g][kb][lane]);
                    t = fmaxf(fmaxf(vm.x, vm.y), fmaxf(vm.z, vm.w));
                }
                const bool need = lane < kRows && t > r_l + kHeadroom;
                if (__ballot_sync(0xffffffffu, need)) {
                    const float rn = need ? t - ref_shift : r_l;
                    const float a = need ? exp2f(r_l - rn) : 1.f;  // r_l = -inf: nothing to keep
                    r_l = rn;
                    if (p.test_counts && quad == 0 && lane == 0) {
                        atomicAdd(p.test_counts + 1, 1);
                        if (k > 0) atomicAdd(p.test_counts, 1);
                    }
#pragma unroll
                    for (int j = 0; j < kHL; ++j) {
                        rr[j] = __shfl_sync(0xffffffffu, rn, kHL * half + j);
                        lp[j] *= __shfl_sync(0xffffffffu, a, kHL * half + j);
                    }
                    if (k > 0) {  // the accumulated tile is rescaled below
                        rescale = true;
                        a_mv = a;
                    }
                }
            }
            // ---- probabilities of this page -> [p1 | p2] operand ----
            // Buffer kb was last read by this group's PV two pages ago.
            if (!fail && k >= 2) fail = !warp_wait(&S.pv_done[g][kb], ((k >> 1) - 1) & 1, abort, p.err);
            if (!fail) {
#pragma unroll
                for (int j = 0; j < kHL; ++j) {
                    s[j] = (s[j] == NEG) ? 0.f : exp2f(s[j] - rr[j]);
                    lp[j] += s[j];
                }
                {
                    // 8 bytes of p1 codes and 8 of p2 codes: heads 8*half .. 8*half + 7
                    uint32_t w1[2] = {0, 0}, w2[2] = {0, 0};
#pragma unroll
                    for (int j = 0; j < kHL; j += 2) {
                        uint32_t c1, c2;
                        split_p(s[j], s[j + 1], c1, c2);
                        w1[j >> 2] |= (c1 & 0xffffu) << (8 * (j & 3));
                        w2[j >> 2] |= (c2 & 0xffffu) << (8 * (j & 3));
                    }
                    uint8_t* pp = S.pp[g][kb];
                    *reinterpret_cast<uint2*>(pp + pp_off(kHL * half, pr)) = make_uint2(w1[0], w1[1]);
                    *reinterpret_cast<uint2*>(pp + pp_off(kNq + kHL * half, pr)) = make_uint2(w2[0], w2[1]);
                    // Rows past the partition's end (or of a page whose id was out of
                    // range) may hold anything, even NaN codes: zero them so that
                    // 0 * x stays 0 in the PV product.
                    if (half == 0 && (!page_ok || pos >= p_end)) {
                        uint8_t* row = S.slot[i % kStages] + pr * 64;
#pragma unroll
                        for (int j = 0; j < kBoxes; ++j) {
                            uint4* q4 = reinterpret_cast<uint4*>(row + j * kBoxBytes);
                            q4[0] = q4[1] = q4[2] = q4[3] = make_uint4(0, 0, 0, 0);
                        }
                    }
                }
                if (rescale) {
                    // The tile holds PV of this group's pages 0..k-1: wait for the
                    // last of them (the probabilities above overlapped that wait),
                    // then scale every head's columns.
                    if (!warp_wait(&S.pv_done[g][(k - 1) & 1], ((k - 1) >> 1) & 1, abort, p.err)) {
                        fail = true;
                    } else {
                        tc_fence_after();
#pragma unroll
                        for (int c = 0; c < 4; ++c) {
                            uint32_t v[32];
                            tmem_ld32(to + 32 * c, v);
                            tmem_wait_ld();
#pragma unroll
                            for (int j = 0; j < 32; ++j) {
                                const float al = __shfl_sync(0xffffffffu, a_mv, j & 15);  // lane h: head h
                                if ((j & 15) < kRows) v[j] = __float_as_uint(__uint_as_float(v[j]) * al);
                            }
                            tmem_st32(to + 32 * c, v);
                        }
                        tmem_wait_st();
                    }
                }
                if (!fail) {
                    fence_async_smem();
                    tc_fence_before();  // TMEM stores of a rescale precede the next PV
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&S.p_full[g][kb]);
                }
            }
        }

        // ---- the group's accumulated tile is complete once its last PV is ----
        const int cnt = n_pages > g ? (n_pages - g + kGroups - 1) / kGroups : 0;
        bool o_ok = !fail && cnt > 0;
        if (o_ok) o_ok = warp_wait(&S.pv_done[g][(cnt - 1) & 1], ((cnt - 1) >> 1) & 1, abort, p.err);
        const float m_run = r_l;

        // ---- this group's normaliser: reduce the per-thread partials ----
        {
            float e[kNq];
#pragma unroll
            for (int h = 0; h < kNq; ++h) e[h] = (h < kRows && (h >> 3) == half) ? lp[h & 7] : 0.f;
            const float wsum = warp_transpose_reduce<false>(e, lane);
            if ((lane & 1) == 0) S.red_l[g][lane >> 1][quad] = wsum;
            __syncwarp();
            if (lane == 0) mbar_arrive(&S.fin_l_bar[g]);
        }
        const bool l_ok = __all_sync(0xffffffffu, wait_bounded(&S.fin_l_bar[g], 0, abort, p.err));
        float l_run = 0.f;  // lane h: normaliser of head h
        if (lane < kNq && l_ok) {
            const float4 vl = *reinterpret_cast<const float4*>(S.red_l[g][lane]);
            l_run = (vl.x + vl.y) + (vl.z + vl.w);
        }

        // ---- combine the warpgroups' states; write the answer ----
        // The warpgroup that owns the partition's last page finishes last.  The
        // other one publishes its references and normalisers and leaves its
        // tile in TMEM; the last one reads both tiles (its warps see the same
        // TMEM lanes in both) 32 columns at a time and stores the answer rows
        // straight to global memory.
        static_assert(kGroups == 2, "the hand-over assumes two warpgroups");
        const int gc = (n_pages - 1) % kGroups;  // combining warpgroup (n_pages >= 1 here)
        const int gp = 1 - gc;                   // the other one
        const int cnt_p = n_pages > gp ? (n_pages - gp + kGroups - 1) / kGroups : 0;
        if (g == gp) {
            if (quad == 0 && lane < kNq) {
                S.fin[0][lane] = m_run;
                S.fin[1][lane] = l_run;
            }
            if (!o_ok && cnt > 0 && lane == 0) S.fin_bad = 1;  // its tile is not to be read
            tc_fence_before();
            __threadfence_block();
            asm volatile("bar.arrive 4, 256;" ::: "memory");  // state published, tile complete
        } else {
            asm volatile("bar.sync 4, 256;" ::: "memory");
            tc_fence_after();
            const bool other_ok = cnt_p > 0 && S.fin_bad == 0;
            const bool direct = p.n_splits == 1;
            // lane h: the weight of each tile (normaliser and kv_scale folded in)
            float w_own = 0.f, w_park = 0.f;
            if (lane < kNq) {
                const float mp = S.fin[0][lane], lq = S.fin[1][lane];
                const float mn = fmaxf(m_run, mp);
                float l = 0.f;
                if (mn != NEG) {
                    w_own = exp2f(m_run - mn);
                    w_park = exp2f(mp - mn);
                    l = l_run * w_own + lq * w_park;
                }
                const float inv = (l > 0.f) ? kv_scale / l : 0.f;
                w_own *= inv;
                w_park *= inv;
                if (quad == 0 && lane < HTc) {
                    const float lse = (l > 0.f) ? (mn + log2f(l)) * kLn2 : -INFINITY;
                    const int64_t grow = (int64_t)b * HT + lane;
                    if (direct) {
                        if (p.lse) p.lse[grow] = lse;
                    } else {
                        p.part_lse[(int64_t)split * p.B * HT + grow] = lse;
                    }
                }
            }
            const int64_t row0 = (int64_t)b * HT;  // this CTA's first answer row
            const uint32_t tp = tmem + (static_cast<uint32_t>(32 * quad) << 16) + kOCol0 + 128 * gp;
#pragma unroll 1
            for (int c = 0; c < 4; ++c) {
                // O = D(p1) + D(p2) / 16 of each tile, weighted
                float v[kRows];
                uint32_t t[32];
                if (o_ok) {
                    tmem_ld32(to + 32 * c, t);
                    tmem_wait_ld();
                }
#pragma unroll
                for (int h = 0; h < kRows; ++h) {
                    const float wo = __shfl_sync(0xffffffffu, w_own, h);
                    v[h] = o_ok ? fmaf(__uint_as_float(t[16 + h]), 0.0625f, __uint_as_float(t[h])) * wo : 0.f;
                }
                if (other_ok) {
                    tmem_ld32(tp + 32 * c, t);
                    tmem_wait_ld();
#pragma unroll
                    for (int h = 0; h < kRows; ++h) {
                        const float wp = __shfl_sync(0xffffffffu, w_park, h);
                        v[h] = fmaf(fmaf(__uint_as_float(t[16 + h]), 0.0625f, __uint_as_float(t[h])), wp, v[h]);
                    }
                }
#pragma unroll
                for (int h = 0; h < kRows; ++h) {
                    if (h < HTc) {
                        const int64_t at = (row0 + h) * kDv + 128 * c + d;
                        if (direct)
                            p.out[at] = __bfloat16_as_ushort(__float2bfloat16_rn(v[h]));
                        else
                            p.part_out[(int64_t)split * p.B * HT * kDv + at] = v[h];
                    }
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    return true;
}

template <int kRows, bool kLpt>
__global__ void __launch_bounds__(kThreads, 1)
    tc_decode_kernel(const __grid_constant__ CUtensorMap tmap, const __grid_constant__ CUtensorMap tmap_box,
                     const __grid_constant__ DecodeParams p) {
    extern __shared__ uint8_t smem_raw[];
    Smem& S = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int tid = threadIdx.x, warp = tid >> 5;
    // Launched as a programmatic dependent of the previous kernel on the stream:
    // everything before this point overlaps its tail; nothing is read before it.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    bool tmem_held;  // the unit had pages (its set-up allocated TMEM)
    if constexpr (!kLpt) {
        // one CTA per (partition, request) unit
        tmem_held = decode_unit<kRows>(&tmap, &tmap_box, p, S, blockIdx.y, blockIdx.x, -1);
    } else {
        // More units than SMs: CTA k (in launch order) takes entry k of the
        // longest-first order (lpt_order_kernel); past the last unit with
        // history there is nothing to do.
        const int k = blockIdx.y * gridDim.x + blockIdx.x;
        const int2 u = p.lpt_order[k];
        tmem_held = u.x >= 0 && decode_unit<kRows>(&tmap, &tmap_box, p, S, u.x / p.n_splits, u.x % p.n_splits, u.y);
    }
    if (warp == 1 && tmem_held) {
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(S.tmem_base), "r"(kTmemCols)
                     : "memory");
    }
}

// ---------------------------------------------------------------- host side

}  // namespace

static PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn() {
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

// Two views of the cache for the TMA unit.
//  * 3-D byte tensor (64-byte column offset, row = page * 64 + position, 64-byte
//    chunk of the 576-byte row), strides 576 B (row) and 64 B (chunk): one box
//    {64, 64, 9} is a whole page, landing in shared memory as nine 64-position x
//    64-byte tiles (chunk-major) with 64-byte swizzle -- the UMMA SWIZZLE_64B
//    K-major layout of each 64-dim slice of the page.
//  * 2-D byte tensor [rows][576] with 64 x 64-byte boxes and the same swizzle:
//    the same nine tiles as nine copies.
cudaError_t encode_cache_maps(CUtensorMap* map3, CUtensorMap* map2, const uint8_t* kv, int64_t num_pages) {
    auto fn = get_encode_fn();
    if (!fn) return cudaErrorNotSupported;
    const cuuint64_t rows = static_cast<cuuint64_t>(num_pages * kPage);
    {
        cuuint64_t dims[3] = {64, rows, static_cast<cuuint64_t>(kBoxes)};
        cuuint64_t strides[2] = {static_cast<cuuint64_t>(kDqk), 64};
        cuuint32_t box[3] = {64, static_cast<cuuint32_t>(kPage), static_cast<cuuint32_t>(kBoxes)};
        cuuint32_t estr[3] = {1, 1, 1};
        CUresult r = fn(map3, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<uint8_t*>(kv), dims, strides, box,
                        estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    }
    {
        cuuint64_t dims[2] = {static_cast<cuuint64_t>(kDqk), rows};
        cuuint64_t strides[1] = {static_cast<cuuint64_t>(kDqk)};
        cuuint32_t box[2] = {64, static_cast<cuuint32_t>(kPage)};
        cuuint32_t estr[2] = {1, 1};
        CUresult r = fn(map2, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(kv), dims, strides, box,
                        estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    }
    return cudaSuccess;
}

cudaError_t launch_tc_wide(const DecodeParams& p, const CUtensorMap& map, const CUtensorMap& map_box, bool lpt,
                           cudaStream_t stream);

// The smallest shift S in [4, 7] with positions <= 2^(S + 6): the n positions
// one warpgroup accumulates then lose at most n * 2^-(14 + S) <= 2^-8 of the
// row's largest weight to e4m3's subnormal floor.
float reference_shift(long long positions) {
    const double s = std::log2(static_cast<double>(positions > 1 ? positions : 1)) - 6.0;
    return static_cast<float>(s < 4.0 ? 4.0 : (s > 7.0 ? 7.0 : s));
}

bool tc_supports(const DecodeParams& p, int cc_major, int cc_minor) {
    return cc_major == 10 && cc_minor == 3 && p.H * p.T <= kMaxRowsTc && p.num_pages >= 1 &&
           p.num_pages * kPage < (1ll << 31);
}

cudaError_t launch_tc_decode(const DecodeParams& p, cudaStream_t stream, bool* handled) {
    *handled = false;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    static int cc[64][2];
    static int sms[64];
    static bool cc_ready[64];
    static std::mutex mu;
    {
        std::lock_guard<std::mutex> lk(mu);
        if (dev < 0 || dev >= 64) return cudaSuccess;
        if (!cc_ready[dev]) {
            if ((e = cudaDeviceGetAttribute(&cc[dev][0], cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess)
                return e;
            if ((e = cudaDeviceGetAttribute(&cc[dev][1], cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess)
                return e;
            if ((e = cudaDeviceGetAttribute(&sms[dev], cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
                return e;
            for (auto fn : {tc_decode_kernel<12, false>, tc_decode_kernel<16, false>, tc_decode_kernel<12, true>,
                            tc_decode_kernel<16, true>})
                if ((e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                              (int)sizeof(Smem) + 1024)) != cudaSuccess)
                    return e;
            cc_ready[dev] = true;
        }
    }
    if (!tc_supports(p, cc[dev][0], cc[dev][1])) return cudaSuccess;

    // The two maps depend only on the cache's address and page count; a
    // serving loop passes the same cache every step, so keep the last pair
    // this thread encoded (addresses are unique across devices).
    thread_local const uint8_t* map_kv = nullptr;
    thread_local int64_t map_pages = -1;
    thread_local CUtensorMap map, map_box;
    if (p.kv != map_kv || p.num_pages != map_pages) {
        map_kv = nullptr;
        if ((e = encode_cache_maps(&map, &map_box, p.kv, p.num_pages)) != cudaSuccess) return e;
        map_kv = p.kv;
        map_pages = p.num_pages;
    }
    const int HT = p.H * p.T;
    DecodeParams q = p;
    // A warpgroup of the 12-head kernel accumulates every other page of a
    // partition; one of the wide kernel every page (for its rows).
    q.ref_shift = reference_shift(64ll * (HT > kNq ? p.chunk_pages : (p.chunk_pages + 1) / 2));
    // Programmatic dependent launch: the CTAs may be scheduled while the
    // previous kernel on the stream drains; the kernel waits for it
    // (griddepcontrol.wait) before reading anything.
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    // More CTAs than SMs (a batch of many, uneven requests): the CTAs take the
    // units in longest-first order (lpt_order_kernel, launched first) instead of
    // request order.
    auto launch_order = [&]() {
        cudaLaunchConfig_t ocfg = {};
        ocfg.gridDim = dim3(1);
        ocfg.blockDim = dim3(kLptThreads);
        ocfg.stream = stream;
        ocfg.attrs = attr;
        ocfg.numAttrs = 1;
        return cudaLaunchKernelEx(&ocfg, lpt_order_kernel, q);
    };
    const long long units = (long long)p.n_splits * p.B;
    if (HT > kNq) {
        // More than 16 rows: the wide kernel, ceil(H*T / 32) CTAs per
        // (partition, request) with the rows shared evenly.
        q.row_ctas = (HT + kWideRows - 1) / kWideRows;
        q.rows_per_cta = (HT + q.row_ctas - 1) / q.row_ctas;
        const bool lpt = p.n_splits > 1 && p.B <= kLptMaxB && units * q.row_ctas > sms[dev];
        if (lpt && (e = launch_order()) != cudaSuccess) return e;
        e = launch_tc_wide(q, map, map_box, lpt, stream);
        if (e == cudaSuccess) *handled = true;
        return e;
    }
    const bool lpt = p.n_splits > 1 && p.B <= kLptMaxB && units > sms[dev];
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(p.n_splits), static_cast<unsigned>(p.B));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = sizeof(Smem) + 1024;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    // the longest-first order, then the decode (a programmatic dependent of it)
    if (lpt && (e = launch_order()) != cudaSuccess) return e;
    if (lpt)
        e = HT <= 12 ? cudaLaunchKernelEx(&cfg, tc_decode_kernel<12, true>, map, map_box, q)
                     : cudaLaunchKernelEx(&cfg, tc_decode_kernel<16, true>, map, map_box, q);
    else
        e = HT <= 12 ? cudaLaunchKernelEx(&cfg, tc_decode_kernel<12, false>, map, map_box, q)
                     : cudaLaunchKernelEx(&cfg, tc_decode_kernel<16, false>, map, map_box, q);
    if (e != cudaSuccess) return e;
    e = cudaGetLastError();
    if (e == cudaSuccess) *handled = true;
    return e;
}

}  // namespace mla
