// mla_tc.cu -- tcgen05 tensor-core split-KV MLA decode over a paged FP8 latent
// cache, for sm_103a (GB300).
//
// Method: "Kimi K3 on AMD Instinct MI355X" post -- section 4 (the history is
// cut into parallel partitions inside one GPU and the partial results are
// combined; KV storage is unchanged), section 1 (each partial answer carries
// its log-sum-exp so partials merge exactly), benchmark section (FP8 KV).
//
// Design (GB300-first):
//   * The FP8 codes are MMA operands as they sit in the cache: every 64-position
//     page is bulk-copied by TMA (nine 64x64-byte boxes, 64-byte swizzle) into a
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
//   * Probabilities are scaled per tile: P = 2^(s - m_tile) in [0, 1], stored as
//     two e4m3 terms p1 + p2 / 16 of 256 * P (relative error ~2^-8, the bf16
//     level); the running output, max and normaliser live in registers of the
//     correction warps and absorb each tile with exact fp32 LSE rescaling.
//   * Warp roles: warp 0 TMA producer, warp 1 TMEM owner + MMA issuer, warps 4-7
//     softmax (TMEM lanes of the score tile), warps 8-11 correction/epilogue
//     (TMEM lanes = latent dims).  Every wait is bounded; on timeout the kernel
//     records an error, drains its own copies and MMAs, frees TMEM and returns.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include <mutex>

#include "mla_internal.cuh"

namespace mla {
namespace {

constexpr int kThreads = 384;
constexpr int kStages = 5;                   // page slots in the TMA ring
constexpr int kNq = 16;                      // rows (t, h) per CTA, padded
constexpr int kNqk = 2 * kNq;                // MMA N: q1 rows | q2 rows (and p1 | p2)
constexpr int kSlotBytes = kPage * kDqk;     // 36,864: one page
constexpr int kBoxBytes = kPage * 64;        // 4,096: 64 positions x 64 dims
constexpr int kBoxes = kDqk / 64;            // 9
constexpr int kQpBytes = kNqk * kDqk;        // 18,432
constexpr int kPpBytes = kNqk * kPage;       // 2,048
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kSCol0 = 0;               // S buffers: cols [0,32) and [32,64)
constexpr uint32_t kOCol0 = 64;              // O buffers: cols [64,192) and [192,320)
constexpr unsigned long long kTimeoutNs = 2000000000ull;  // 2 s per wait

struct Smem {
    uint8_t slot[kStages][kSlotBytes];       // 1024-aligned page tiles
    uint8_t qp[kQpBytes];                    // [q1 | q2] K-major, no swizzle
    uint8_t pp[2][kPpBytes];                 // [p1 | p2] K-major, no swizzle
    float red_m[2][kNq][4];                  // per-warp tile maxima (softmax)
    float red_l[2][kNq][4];                  // per-warp tile sums (-> correction)
    float stat_m[2][kNq];                    // tile maxima (-> correction)
    float row_scale[kNq];                    // kv_scale * sm_scale * log2(e) * 2^-e
    int rowlim[kNq];                         // visible prefix per row; -1 = padding
    uint64_t full[kStages], empty[kStages];
    uint64_t s_full[2], s_empty[2], p_full[2], o_full[2], o_empty[2], red_bar[2];
    uint64_t mma_done;
    uint32_t tmem_base;
    int abort;
};
static_assert(sizeof(uint8_t[kStages][kSlotBytes]) % 1024 == 0, "slots keep 1 KB alignment");

// ---------------------------------------------------------------- PTX wrappers

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Wait for the phase of `parity` to complete, giving up after kTimeoutNs or
// when another role has aborted.  Returns false on give-up.
__device__ __forceinline__ bool wait_bounded(uint64_t* bar, uint32_t parity, volatile int* abort, int* err) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 127u) == 0) {
            if (*abort) return false;
            if (global_ns() - t0 > kTimeoutNs) {
                *abort = 1;
                atomicCAS(err, 0, kErrWaitTimeout);
                return false;
            }
        }
    }
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Shared-memory matrix descriptor (tcgen05): start, leading / stride byte
// offsets, version 1, layout type (0 none, 4 = 64-byte swizzle).
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo,
                                              uint32_t layout) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
    d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
    d |= static_cast<uint64_t>(1) << 46;
    d |= static_cast<uint64_t>(layout & 7u) << 61;
    return d;
}
constexpr uint32_t kLayoutNone = 0;
constexpr uint32_t kLayoutSw64 = 4;

// Instruction descriptor, kind::f8f6f4, A = B = e4m3, D = f32.
__host__ __device__ constexpr uint32_t idesc_e4m3(int M, int N, bool a_mn_major, bool b_mn_major) {
    return (1u << 4) | ((a_mn_major ? 1u : 0u) << 15) | ((b_mn_major ? 1u : 0u) << 16) |
           (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}
constexpr uint32_t kIdescQK = idesc_e4m3(64, kNqk, false, false);
constexpr uint32_t kIdescPV = idesc_e4m3(128, kNqk, true, false);

__device__ __forceinline__ void mma_e4m3(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                         uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// e4m3 helpers (round to nearest even, saturating to +-448)
__device__ __forceinline__ uint32_t f2_to_e4m3x2(float a, float b) {
    return static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3));
}
__device__ __forceinline__ float2 e4m3x2_to_f2(uint32_t v) {
    __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(v & 0xffffu), __NV_E4M3);
    return __half22float2(*reinterpret_cast<__half2*>(&h));
}

// Byte offset of element (row n, k) in a K-major, no-swizzle operand made of
// 8-row x 16-byte core matrices: LBO = 128 B along K, SBO = (K/16) * 128 along rows.
__device__ __forceinline__ uint32_t kmajor_off(int n, int k, int K) {
    return (n & 7) * 16 + (n >> 3) * (K / 16) * 128 + (k & 15) + (k >> 4) * 128;
}

// Transpose-reduce: 16 values per lane across the 32 lanes of a warp.  On
// return v[0] of lane l holds the reduction of value index l >> 1.
template <bool kMax>
__device__ __forceinline__ float warp_transpose_reduce(float (&v)[16], int lane) {
#pragma unroll
    for (int w = 8, sh = 16; w >= 1; w >>= 1, sh >>= 1) {
        const bool hi = (lane & sh) != 0;
#pragma unroll
        for (int i = 0; i < w; ++i) {
            const float send = hi ? v[i] : v[i + w];
            const float keep = hi ? v[i + w] : v[i];
            const float recv = __shfl_xor_sync(0xffffffffu, send, sh);
            v[i] = kMax ? fmaxf(keep, recv) : keep + recv;
        }
    }
    const float other = __shfl_xor_sync(0xffffffffu, v[0], 1);
    return kMax ? fmaxf(v[0], other) : v[0] + other;
}

__global__ void __launch_bounds__(kThreads, 1)
    tc_decode_kernel(const __grid_constant__ CUtensorMap tmap, const DecodeParams p) {
    extern __shared__ uint8_t smem_raw[];
    Smem& S = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int split = blockIdx.x, b = blockIdx.y;
    const int HT = p.H * p.T;
    volatile int* abort = &S.abort;

    int L = __ldg(p.seq_lens + b);
    if (L < 0 || L > p.max_pages * kPage || (L > 0 && L < p.T)) {
        if (tid == 0) atomicCAS(p.err, 0, kErrSeqRange);
        L = 0;
    }
    const int p_begin = split * p.chunk_pages * kPage;
    const int p_end = min(L, p_begin + p.chunk_pages * kPage);
    const int pg_begin = p_begin / kPage;
    const int n_pages = p_end > p_begin ? (p_end - p_begin + kPage - 1) / kPage : 0;
    const float kv_scale = __ldg(p.kv_scale);

    // ---------------- set-up: barriers, TMEM, query operand ----------------
    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&S.full[s], 1);
            mbar_init(&S.empty[s], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&S.s_full[i], 1);
            mbar_init(&S.s_empty[i], 4);
            mbar_init(&S.p_full[i], 4);
            mbar_init(&S.o_full[i], 1);
            mbar_init(&S.o_empty[i], 4);
            mbar_init(&S.red_bar[i], 4);
        }
        mbar_init(&S.mma_done, 1);
        S.abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(&S.tmem_base)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    // Query rows: warp w prepares rows w and w + 12 (< 16).
    for (int r = warp; r < kNq; r += kThreads / 32) {
        if (r < HT) {
            const uint4* src = reinterpret_cast<const uint4*>(p.q + ((int64_t)b * HT + r) * kDqk);
            uint4 v[3];
            float amax = 0.f;
#pragma unroll
            for (int k = 0; k < 3; ++k) {
                const int c = lane + 32 * k;  // 16-byte chunk: 8 bf16 values
                v[k] = c < kDqk / 8 ? __ldg(src + c) : make_uint4(0, 0, 0, 0);
                const uint32_t w[4] = {v[k].x, v[k].y, v[k].z, v[k].w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    amax = fmaxf(amax, fabsf(__uint_as_float(w[j] << 16)));
                    amax = fmaxf(amax, fabsf(__uint_as_float(w[j] & 0xffff0000u)));
                }
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
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
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = S.tmem_base;
    asm volatile("griddepcontrol.launch_dependents;");

    if (warp == 0) {
        // ======================= TMA producer =======================
        if (lane == 0 && n_pages > 0) {
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap)) : "memory");
            int issued = 0;
            for (int i = 0; i < n_pages; ++i) {
                const int s = i % kStages;
                if (!wait_bounded(&S.empty[s], ((i / kStages) & 1) ^ 1, abort, p.err)) break;
                int32_t pid = __ldg(p.block_table + (int64_t)b * p.bt_stride + pg_begin + i);
                if (pid < 0 || pid >= p.num_pages) {
                    atomicCAS(p.err, 0, kErrPageRange);
                    pid = 0;  // load a valid page; the softmax masks and zeroes it
                }
                mbar_expect_tx(&S.full[s], kSlotBytes);
                const uint32_t dst = smem_u32(S.slot[s]);
#pragma unroll
                for (int j = 0; j < kBoxes; ++j)
                    tma_load_2d(dst + j * kBoxBytes, &tmap, 64 * j, pid * kPage, &S.full[s]);
                issued = i + 1;
            }
            // Drain: never leave with a copy in flight into this CTA's shared memory.
            for (int i = max(0, issued - kStages); i < issued; ++i) {
                const int s = i % kStages;
                const uint32_t par = (i / kStages) & 1;
                if (mbar_try_wait(&S.full[s], par)) continue;
                const uint64_t t0 = global_ns();
                while (!mbar_try_wait(&S.full[s], par) && global_ns() - t0 < kTimeoutNs) {
                }
            }
        }
    } else if (warp == 1) {
        // ======================= MMA issuer =======================
        if (lane == 0 && n_pages > 0) {
            const uint32_t qp = smem_u32(S.qp);
            auto issue_qk = [&](int i) -> bool {
                const int s = i % kStages, buf = i & 1;
                if (!wait_bounded(&S.full[s], (i / kStages) & 1, abort, p.err)) return false;
                if (!wait_bounded(&S.s_empty[buf], ((i >> 1) & 1) ^ 1, abort, p.err)) return false;
                tc_fence_after();
                const uint32_t slot = smem_u32(S.slot[s]);
                const uint32_t d = tmem + kSCol0 + 32 * buf;
#pragma unroll
                for (int ks = 0; ks < kDqk / 32; ++ks) {
                    const uint64_t a = smem_desc(slot + (ks >> 1) * kBoxBytes + (ks & 1) * 32, 16, 512,
                                                 kLayoutSw64);
                    const uint64_t bd = smem_desc(qp + ks * 256, 128, (kDqk / 16) * 128, kLayoutNone);
                    mma_e4m3(d, a, bd, kIdescQK, ks > 0);
                }
                mma_commit(&S.s_full[buf]);
                return true;
            };
            bool ok = issue_qk(0);
            for (int i = 0; ok && i < n_pages; ++i) {
                if (i + 1 < n_pages && !(ok = issue_qk(i + 1))) break;
                const int s = i % kStages, buf = i & 1;
                if (!wait_bounded(&S.p_full[buf], (i >> 1) & 1, abort, p.err)) break;
                if (!wait_bounded(&S.o_empty[buf], ((i >> 1) & 1) ^ 1, abort, p.err)) break;
                tc_fence_after();
                const uint32_t slot = smem_u32(S.slot[s]);
                const uint32_t pp = smem_u32(S.pp[buf]);
#pragma unroll
                for (int c = 0; c < kDv / 128; ++c) {
#pragma unroll
                    for (int ks = 0; ks < kPage / 32; ++ks) {
                        const uint64_t a = smem_desc(slot + 2 * c * kBoxBytes + ks * 32 * 64, kBoxBytes,
                                                     512, kLayoutSw64);
                        const uint64_t bd = smem_desc(pp + ks * 256, 128, (kPage / 16) * 128, kLayoutNone);
                        mma_e4m3(tmem + kOCol0 + 128 * buf + 32 * c, a, bd, kIdescPV, ks > 0);
                    }
                }
                mma_commit(&S.o_full[buf]);
                mma_commit(&S.empty[s]);
            }
            // Drain: every MMA this thread issued completes before TMEM is freed.
            mma_commit(&S.mma_done);
            const uint64_t t0 = global_ns();
            while (!mbar_try_wait(&S.mma_done, 0) && global_ns() - t0 < kTimeoutNs) {
            }
        }
    } else if (warp >= 4 && warp < 8) {
        // ======================= softmax =======================
        // Every hand-off goes through an mbarrier with a bounded wait (no named
        // barriers), so a role that gives up can never leave another one blocked.
        const int sw = warp - 4;                 // TMEM lane quadrant
        const bool has_row = lane < 16;          // M=64 score tile: 16 rows per quadrant
        const int pr = 16 * sw + lane;           // position within the page
        const float NEG = -INFINITY;
        for (int i = 0; i < n_pages; ++i) {
            const int buf = i & 1;
            if (!__all_sync(0xffffffffu, wait_bounded(&S.s_full[buf], (i >> 1) & 1, abort, p.err))) break;
            tc_fence_after();
            uint32_t r1[16], r2[16];
            const uint32_t ta = tmem + (static_cast<uint32_t>(32 * sw) << 16) + kSCol0 + 32 * buf;
            tmem_ld16(ta, r1);
            tmem_ld16(ta + 16, r2);
            tmem_wait_ld();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&S.s_empty[buf]);

            const int pg = pg_begin + i;
            const int32_t pid = __ldg(p.block_table + (int64_t)b * p.bt_stride + pg);
            const bool page_ok = pid >= 0 && pid < p.num_pages;
            const int pos = pg * kPage + pr;
            const bool in_part = has_row && page_ok && pos < p_end;
            float s[kNq], e[kNq];
#pragma unroll
            for (int h = 0; h < kNq; ++h) {
                const float v = (__uint_as_float(r1[h]) + __uint_as_float(r2[h]) * 0.0625f) * S.row_scale[h];
                s[h] = (in_part && pos < S.rowlim[h]) ? v : NEG;
                e[h] = s[h];
            }
            const float wmax = warp_transpose_reduce<true>(e, lane);
            if ((lane & 1) == 0) S.red_m[buf][lane >> 1][sw] = wmax;
            __syncwarp();
            if (lane == 0) mbar_arrive(&S.red_bar[buf]);
            if (!__all_sync(0xffffffffu, wait_bounded(&S.red_bar[buf], (i >> 1) & 1, abort, p.err))) break;
            float m[kNq];
#pragma unroll
            for (int h = 0; h < kNq; ++h) {
                const float4 v = *reinterpret_cast<const float4*>(S.red_m[buf][h]);
                m[h] = fmaxf(fmaxf(v.x, v.y), fmaxf(v.z, v.w));
                e[h] = (s[h] == NEG) ? 0.f : exp2f(s[h] - m[h]);
                s[h] = e[h];  // keep the probabilities; e is consumed by the sum
            }
            const float wsum = warp_transpose_reduce<false>(e, lane);
            // P and the statistics of buffer `buf` were last used by tile i - 2.
            if (i >= 2 &&
                !__all_sync(0xffffffffu, wait_bounded(&S.o_empty[buf], ((i >> 1) & 1) ^ 1, abort, p.err)))
                break;
            if ((lane & 1) == 0) {
                S.red_l[buf][lane >> 1][sw] = wsum;
                if (sw == 0) {
                    const float4 v = *reinterpret_cast<const float4*>(S.red_m[buf][lane >> 1]);
                    S.stat_m[buf][lane >> 1] = fmaxf(fmaxf(v.x, v.y), fmaxf(v.z, v.w));
                }
            }
            if (has_row) {
                uint8_t* pp = S.pp[buf];
#pragma unroll
                for (int h = 0; h < kNq; h += 2) {
                    const float a0 = s[h] * 256.f, a1 = s[h + 1] * 256.f;
                    const uint32_t c1 = f2_to_e4m3x2(a0, a1);
                    const float2 back = e4m3x2_to_f2(c1);
                    const uint32_t c2 = f2_to_e4m3x2((a0 - back.x) * 16.f, (a1 - back.y) * 16.f);
                    pp[kmajor_off(h, pr, kPage)] = static_cast<uint8_t>(c1 & 0xff);
                    pp[kmajor_off(h + 1, pr, kPage)] = static_cast<uint8_t>(c1 >> 8);
                    pp[kmajor_off(kNq + h, pr, kPage)] = static_cast<uint8_t>(c2 & 0xff);
                    pp[kmajor_off(kNq + h + 1, pr, kPage)] = static_cast<uint8_t>(c2 >> 8);
                }
                // Rows past the partition's end (or of a page whose id was out of
                // range) may hold anything, even NaN codes: zero them so that
                // 0 * x stays 0 in the PV product.
                if (!page_ok || pos >= p_end) {
                    uint8_t* row = S.slot[i % kStages] + pr * 64;
#pragma unroll
                    for (int j = 0; j < kBoxes; ++j) {
                        uint4* q4 = reinterpret_cast<uint4*>(row + j * kBoxBytes);
                        q4[0] = q4[1] = q4[2] = q4[3] = make_uint4(0, 0, 0, 0);
                    }
                }
            }
            fence_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&S.p_full[buf]);
        }
    } else if (warp >= 8) {
        // ======================= correction + epilogue =======================
        // Thread (warp 8 + cw, lane) owns latent dims 32*cw + lane of each 128-dim
        // block.  The running max / normaliser of head h is identical in every
        // thread: lane h of each warp keeps it and broadcasts it by shuffle.
        const int cw = warp - 8;
        const int d = 32 * cw + lane;
        float o[4][kNq];
        float m_run = -INFINITY, l_run = 0.f;    // lane h < 16: head h
#pragma unroll
        for (int h = 0; h < kNq; ++h)
#pragma unroll
            for (int c = 0; c < 4; ++c) o[c][h] = 0.f;
        for (int i = 0; i < n_pages; ++i) {
            const int buf = i & 1;
            if (!__all_sync(0xffffffffu, wait_bounded(&S.o_full[buf], (i >> 1) & 1, abort, p.err))) break;
            // p_full of this tile has completed (PV waited on it); waiting on it here
            // orders the softmax's statistics writes before the reads below.
            if (!__all_sync(0xffffffffu, wait_bounded(&S.p_full[buf], (i >> 1) & 1, abort, p.err))) break;
            tc_fence_after();
            float a_l = 1.f, b_l = 0.f;
            if (lane < kNq) {
                const float mt = S.stat_m[buf][lane];
                const float4 lp = *reinterpret_cast<const float4*>(S.red_l[buf][lane]);
                const float lt = (lp.x + lp.y) + (lp.z + lp.w);
                const float mn = fmaxf(m_run, mt);
                if (mn != -INFINITY) {
                    a_l = exp2f(m_run - mn);
                    b_l = exp2f(mt - mn);
                    l_run = l_run * a_l + lt * b_l;
                    m_run = mn;
                }
            }
            float alpha[kNq], beta[kNq];
#pragma unroll
            for (int h = 0; h < kNq; ++h) {
                alpha[h] = __shfl_sync(0xffffffffu, a_l, h);
                beta[h] = __shfl_sync(0xffffffffu, b_l, h) * (1.f / 256.f);
            }
            const uint32_t ta = tmem + (static_cast<uint32_t>(32 * cw) << 16) + kOCol0 + 128 * buf;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint32_t r[16];
                tmem_ld16(ta + 32 * c, r);
                tmem_wait_ld();
#pragma unroll
                for (int h = 0; h < kNq; ++h) o[c][h] = fmaf(o[c][h], alpha[h], beta[h] * __uint_as_float(r[h]));
                tmem_ld16(ta + 32 * c + 16, r);
                tmem_wait_ld();
#pragma unroll
                for (int h = 0; h < kNq; ++h) o[c][h] = fmaf(beta[h] * 0.0625f, __uint_as_float(r[h]), o[c][h]);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&S.o_empty[buf]);
        }
        // epilogue: normalised partial answer (or final output) and its LSE
        const bool direct = p.n_splits == 1;
#pragma unroll
        for (int h = 0; h < kNq; ++h) {
            const float l = __shfl_sync(0xffffffffu, l_run, h);
            if (h >= HT) continue;
            const int64_t grow = (int64_t)b * HT + h;
            if (direct) {
                const float inv = (l > 0.f) ? kv_scale / l : 0.f;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    __nv_bfloat16 v = __float2bfloat16_rn(o[c][h] * inv);
                    p.out[grow * kDv + 128 * c + d] = *reinterpret_cast<uint16_t*>(&v);
                }
            } else if (l > 0.f) {
                const float inv = kv_scale / l;
                const int64_t prow = (int64_t)split * p.B * HT + grow;
#pragma unroll
                for (int c = 0; c < 4; ++c) p.part_out[prow * kDv + 128 * c + d] = o[c][h] * inv;
            }
        }
        if (cw == 0 && lane < HT && lane < kNq) {
            const float lse = (l_run > 0.f) ? (m_run + log2f(l_run)) * kLn2 : -INFINITY;
            const int64_t grow = (int64_t)b * HT + lane;
            if (direct) {
                if (p.lse) p.lse[grow] = lse;
            } else {
                p.part_lse[(int64_t)split * p.B * HT + grow] = lse;
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) {
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols)
                     : "memory");
    }
}

// ---------------------------------------------------------------- host side

PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn() {
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

// The cache viewed as a 2-D byte tensor [num_pages * 64 rows][576 cols]; boxes of
// 64 rows x 64 bytes with 64-byte swizzle (the UMMA SWIZZLE_64B atom).
cudaError_t encode_cache_map(CUtensorMap* map, const uint8_t* kv, int64_t num_pages) {
    auto fn = get_encode_fn();
    if (!fn) return cudaErrorNotSupported;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(kDqk), static_cast<cuuint64_t>(num_pages * kPage)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(kDqk)};
    cuuint32_t box[2] = {64, static_cast<cuuint32_t>(kPage)};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(kv), dims, strides, box,
                    estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace

bool tc_supports(const DecodeParams& p, int cc_major, int cc_minor) {
    return cc_major == 10 && cc_minor == 3 && p.H * p.T <= kNq && p.num_pages >= 1 &&
           p.num_pages * kPage < (1ll << 31);
}

cudaError_t launch_tc_decode(const DecodeParams& p, cudaStream_t stream, bool* handled) {
    *handled = false;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    static int cc[64][2];
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
            if ((e = cudaFuncSetAttribute(tc_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          (int)sizeof(Smem) + 1024)) != cudaSuccess)
                return e;
            cc_ready[dev] = true;
        }
    }
    if (!tc_supports(p, cc[dev][0], cc[dev][1])) return cudaSuccess;
    CUtensorMap map;
    if ((e = encode_cache_map(&map, p.kv, p.num_pages)) != cudaSuccess) return e;
    dim3 grid(p.n_splits, p.B);
    tc_decode_kernel<<<grid, kThreads, sizeof(Smem) + 1024, stream>>>(map, p);
    e = cudaGetLastError();
    if (e == cudaSuccess) *handled = true;
    return e;
}

}  // namespace mla
