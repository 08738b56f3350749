// mla_api.cu -- host side of the C ABI declared in include/mla_decode.h:
// argument validation, split planning, library-owned scratch, kernel dispatch
// and error reporting.  Everything here runs on the host; every step of the
// attention itself runs in the CUDA kernels.
#include <algorithm>
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <functional>
#include <map>
#include <mutex>
#include <string>
#include <utility>
#include <vector>

#include "../../include/mla_decode.h"
#include "../../include/mla_decode_testing.h"
#include "mla_host.h"
#include "mla_internal.cuh"

// The device error word written by kernels (bounded waits, bounds checks).
__device__ int g_mla_device_error;

namespace mla {

namespace {

thread_local std::string t_last_error;
thread_local cudaEvent_t t_prof_begin = nullptr;
thread_local cudaEvent_t t_prof_end = nullptr;
thread_local int t_last_impl = 0;
// Test hooks (include/mla_decode_testing.h): per calling thread.
thread_local int* t_test_counts = nullptr;  // one-shot: the next decode call only
thread_local int t_test_stall = 0;
std::atomic<int> g_impl{MLA_IMPL_AUTO};

mla_status_t fail(mla_status_t st, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    t_last_error = buf;
    return st;
}

mla_status_t cuda_fail(cudaError_t e, const char* what) {
    cudaGetLastError();  // clear a sticky launch error so later calls are not blamed
    return fail(MLA_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

// Per-device facts, filled once per device.
struct DeviceInfo {
    bool ready = false;
    int sm_count = 0;
    int* err_word = nullptr;
};
std::mutex g_dev_mu;
DeviceInfo g_dev[64];

mla_status_t device_info(DeviceInfo** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= 64) return fail(MLA_ERR_UNSUPPORTED, "device ordinal %d >= 64", dev);
    std::lock_guard<std::mutex> lk(g_dev_mu);
    DeviceInfo& d = g_dev[dev];
    if (!d.ready) {
        e = cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
        void* addr = nullptr;
        e = cudaGetSymbolAddress(&addr, g_mla_device_error);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(device error word)");
        d.err_word = static_cast<int*>(addr);
        d.ready = true;
    }
    *out = &d;
    return MLA_OK;
}

// Library-owned split scratch, one buffer per (device, stream), grown in
// stream order so that a buffer is never released while a kernel still uses it.
// A buffer that a captured CUDA graph uses is never released at all (the graph
// may be replayed at any later time): growing it retires it instead.  Growing
// during a capture is refused, so a graph never owns a stream-ordered
// allocation of the library.
struct Scratch {
    void* ptr = nullptr;
    size_t bytes = 0;
    bool in_graph = false;  // used by a call made during stream capture
};
std::mutex g_ws_mu;
std::map<std::pair<int, void*>, Scratch> g_ws;
// Buffers a captured call used, kept (with their device) for the graphs that
// may still replay them, until mla_release_graph_scratch.
std::vector<std::pair<int, void*>> g_ws_retired;

mla_status_t get_scratch(size_t need, cudaStream_t stream, void** out) {
    *out = nullptr;
    if (need == 0) return MLA_OK;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    e = cudaStreamIsCapturing(stream, &cap);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamIsCapturing");
    const bool capturing = cap != cudaStreamCaptureStatusNone;
    std::lock_guard<std::mutex> lk(g_ws_mu);
    Scratch& s = g_ws[{dev, static_cast<void*>(stream)}];
    if (s.bytes < need) {
        if (capturing)
            return fail(MLA_ERR_UNSUPPORTED,
                        "the split scratch of this stream must grow to %zu bytes, which cannot happen "
                        "during stream capture: make one uncaptured call of this size on the stream "
                        "first",
                        need);
        if (s.ptr) {
            if (s.in_graph) {
                g_ws_retired.push_back({dev, s.ptr});
            } else {
                e = cudaFreeAsync(s.ptr, stream);
                if (e != cudaSuccess) return cuda_fail(e, "cudaFreeAsync(scratch)");
            }
            s.ptr = nullptr;
            s.bytes = 0;
            s.in_graph = false;
        }
        size_t grow = need + need / 4;
        e = cudaMallocAsync(&s.ptr, grow, stream);
        if (e != cudaSuccess) {
            cudaGetLastError();
            s.ptr = nullptr;
            return fail(MLA_ERR_NO_MEMORY, "cudaMallocAsync(%zu bytes) for split scratch: %s", grow,
                        cudaGetErrorString(e));
        }
        s.bytes = grow;
    }
    if (capturing) s.in_graph = true;
    *out = s.ptr;
    return MLA_OK;
}

bool contiguous(const mla_tensor_t* t) {
    int64_t expect = 1;
    for (int i = t->ndim - 1; i >= 0; --i) {
        if (t->shape[i] != 1 && t->stride[i] != expect) return false;
        expect *= t->shape[i];
    }
    return true;
}

mla_status_t check_tensor(const mla_tensor_t* t, const char* name, int ndim, int dtype,
                          bool need_contig, size_t align) {
    if (!t) return fail(MLA_ERR_INVALID_ARG, "%s: null descriptor", name);
    if (t->ndim != ndim) return fail(MLA_ERR_INVALID_ARG, "%s: rank %d, expected %d", name, t->ndim, ndim);
    if (t->dtype != dtype) return fail(MLA_ERR_INVALID_ARG, "%s: dtype %d, expected %d", name, t->dtype, dtype);
    for (int i = 0; i < ndim; ++i)
        if (t->shape[i] < 0) return fail(MLA_ERR_INVALID_ARG, "%s: negative dim %d", name, i);
    if (need_contig && !contiguous(t))
        return fail(MLA_ERR_UNSUPPORTED, "%s: must be contiguous", name);
    int64_t numel = 1;
    for (int i = 0; i < ndim; ++i) numel *= t->shape[i];
    if (numel > 0 && !t->data) return fail(MLA_ERR_INVALID_ARG, "%s: null data", name);
    if (align > 1 && (reinterpret_cast<uintptr_t>(t->data) % align) != 0)
        return fail(MLA_ERR_UNSUPPORTED, "%s: data must be %zu-byte aligned", name, align);
    return MLA_OK;
}

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

}  // namespace

void internal_carve_scratch(DecodeParams& p, void* ws) {
    const size_t out_bytes = (size_t)p.n_splits * p.B * p.T * p.H * kDv * sizeof(float);
    const size_t lse_bytes = (size_t)p.n_splits * p.B * p.T * p.H * sizeof(float);
    char* base = static_cast<char*>(ws);
    p.part_out = reinterpret_cast<float*>(base);
    p.part_lse = reinterpret_cast<float*>(base + ((out_bytes + 255) & ~size_t(255)));
    p.lpt_order = reinterpret_cast<int2*>(base + ((out_bytes + 255) & ~size_t(255)) + ((lse_bytes + 255) & ~size_t(255)));
}

// Accessors for the library's other host translation units (mla_host.h).
mla_status_t internal_fail(mla_status_t st, const char* msg) { return fail(st, "%s", msg); }
mla_status_t internal_cuda_fail(cudaError_t e, const char* what) { return cuda_fail(e, what); }
void internal_clear_error() { t_last_error.clear(); }
mla_status_t internal_device(int** err_word, int* sm_count) {
    DeviceInfo* d = nullptr;
    mla_status_t st = device_info(&d);
    if (st != MLA_OK) return st;
    *err_word = d->err_word;
    *sm_count = d->sm_count;
    return MLA_OK;
}
mla_status_t internal_check_tensor(const mla_tensor_t* t, const char* name, int ndim, int dtype,
                                   bool need_contig, size_t align) {
    return check_tensor(t, name, ndim, dtype, need_contig, align);
}

mla_status_t internal_prepare_decode(const mla_tensor_t* q, const mla_tensor_t* kv_cache, const float* kv_scale,
                                     const mla_tensor_t* block_table, const mla_tensor_t* seq_lens,
                                     int32_t n_splits, int32_t auto_splits_cap, float sm_scale,
                                     const mla_tensor_t* out, const mla_tensor_t* lse, DecodeParams* pp,
                                     bool* empty) {
    *empty = false;
    mla_status_t st;
    if ((st = check_tensor(q, "q", 4, MLA_DTYPE_BF16, true, 16)) != MLA_OK) return st;
    const int64_t B = q->shape[0], T = q->shape[1], H = q->shape[2];
    if (q->shape[3] != kDqk) return fail(MLA_ERR_UNSUPPORTED, "q: last dim %lld, only 576 is supported", (long long)q->shape[3]);
    if (T < 1 || H < 1) return fail(MLA_ERR_INVALID_ARG, "q: T and H must be >= 1");
    if (H * T > kMaxRows) return fail(MLA_ERR_UNSUPPORTED, "H*T = %lld exceeds %d", (long long)(H * T), kMaxRows);
    if ((st = check_tensor(kv_cache, "kv_cache", 3, MLA_DTYPE_E4M3FN, true, 16)) != MLA_OK) return st;
    if (kv_cache->shape[1] != kPage || kv_cache->shape[2] != kDqk)
        return fail(MLA_ERR_UNSUPPORTED, "kv_cache: must be [num_pages, 64, 576]");
    if (!kv_scale) return fail(MLA_ERR_INVALID_ARG, "kv_scale: null pointer");
    if ((st = check_tensor(block_table, "block_table", 2, MLA_DTYPE_I32, false, 4)) != MLA_OK) return st;
    if (block_table->shape[0] != B) return fail(MLA_ERR_INVALID_ARG, "block_table: first dim must be B");
    const int64_t max_pages = block_table->shape[1];
    if (block_table->stride[1] != 1 || block_table->stride[0] < max_pages)
        return fail(MLA_ERR_UNSUPPORTED, "block_table: rows must be contiguous");
    if ((st = check_tensor(seq_lens, "seq_lens", 1, MLA_DTYPE_I32, true, 4)) != MLA_OK) return st;
    if (seq_lens->shape[0] != B) return fail(MLA_ERR_INVALID_ARG, "seq_lens: must have B entries");
    if ((st = check_tensor(out, "out", 4, MLA_DTYPE_BF16, true, 16)) != MLA_OK) return st;
    if (out->shape[0] != B || out->shape[1] != T || out->shape[2] != H || out->shape[3] != kDv)
        return fail(MLA_ERR_INVALID_ARG, "out: must be [B, T, H, 512]");
    if (lse) {
        if ((st = check_tensor(lse, "lse", 3, MLA_DTYPE_F32, true, 4)) != MLA_OK) return st;
        if (lse->shape[0] != B || lse->shape[1] != T || lse->shape[2] != H)
            return fail(MLA_ERR_INVALID_ARG, "lse: must be [B, T, H]");
    }
    if (n_splits < 0) return fail(MLA_ERR_INVALID_ARG, "n_splits must be >= 0");
    if (max_pages < 1 && B > 0) return fail(MLA_ERR_INVALID_ARG, "block_table: needs >= 1 column");
    if (max_pages > (1 << 24)) return fail(MLA_ERR_UNSUPPORTED, "block_table: more than 2^24 pages per request");
    if (B > 65535) return fail(MLA_ERR_UNSUPPORTED, "B > 65535");
    if (B == 0) {
        *empty = true;
        return MLA_OK;
    }

    DeviceInfo* dev = nullptr;
    if ((st = device_info(&dev)) != MLA_OK) return st;

    int32_t req = n_splits;
    if (req == 0) {
        req = mla_auto_splits((int32_t)B, (int32_t)T, (int32_t)H, (int32_t)max_pages, dev->sm_count);
        if (auto_splits_cap > 0 && req > auto_splits_cap) req = auto_splits_cap;
    }
    const int32_t chunk = mla_split_chunk_pages((int32_t)max_pages, req);
    const int32_t n_eff = (int32_t)ceil_div(max_pages, chunk);

    DecodeParams p{};
    p.q = static_cast<const uint16_t*>(q->data);
    p.kv = static_cast<const uint8_t*>(kv_cache->data);
    p.kv_scale = kv_scale;
    p.block_table = static_cast<const int32_t*>(block_table->data);
    p.seq_lens = static_cast<const int32_t*>(seq_lens->data);
    p.bt_stride = block_table->stride[0];
    p.num_pages = kv_cache->shape[0];
    p.B = (int)B;
    p.T = (int)T;
    p.H = (int)H;
    p.max_pages = (int)max_pages;
    p.n_splits = n_eff;
    p.chunk_pages = chunk;
    p.sm_scale_log2 = sm_scale * kLog2e;
    p.out = static_cast<uint16_t*>(out->data);
    p.lse = lse ? static_cast<float*>(lse->data) : nullptr;
    p.err = dev->err_word;
    *pp = p;
    return MLA_OK;
}

mla_status_t internal_launch_decode(DecodeParams& p, cudaStream_t s) {
    // the calling thread's one-shot requests apply to this call only
    cudaEvent_t ev_begin = t_prof_begin, ev_end = t_prof_end;
    t_prof_begin = t_prof_end = nullptr;
    p.test_counts = t_test_counts;
    t_test_counts = nullptr;
    p.test_stall_copies = t_test_stall;

    const int impl = g_impl.load();
    cudaError_t e = cudaSuccess;
    bool handled = false;
    if (ev_begin && (e = cudaEventRecord(ev_begin, s)) != cudaSuccess)
        return cuda_fail(e, "cudaEventRecord(profile begin)");
    if (impl == MLA_IMPL_AUTO || impl == MLA_IMPL_TCGEN05) {
        e = launch_tc_decode(p, s, &handled);
        if (e != cudaSuccess) return cuda_fail(e, "tcgen05 decode launch");
        if (!handled && impl == MLA_IMPL_TCGEN05)
            return fail(MLA_ERR_UNSUPPORTED, "tcgen05 kernel does not support this shape");
    }
    if (!handled) {
        e = launch_simt_decode(p, s);
        if (e != cudaSuccess) return cuda_fail(e, "decode launch");
    }
    t_last_impl = handled ? MLA_IMPL_TCGEN05 : MLA_IMPL_SIMT;
    if (ev_end && (e = cudaEventRecord(ev_end, s)) != cudaSuccess)
        return cuda_fail(e, "cudaEventRecord(profile end)");
    if (p.n_splits > 1) {
        MergeParams m{};
        m.part_out = p.part_out;
        m.part_lse = p.part_lse;
        m.S = p.n_splits;
        m.rows = (int64_t)p.B * p.T * p.H;
        m.in_bf16 = 0;
        m.out = p.out;
        m.lse = p.lse;
        m.pdl = 1;
        // partitions past a request's history are not written (the longest-first
        // launch never visits them): the combine counts them as empty
        m.seq_lens = p.seq_lens;
        m.rows_per_req = p.T * p.H;
        m.T = p.T;
        m.chunk_pages = p.chunk_pages;
        m.max_pages = p.max_pages;
        e = launch_merge(m, s);
        if (e != cudaSuccess) return cuda_fail(e, "split combine launch");
    }
    return MLA_OK;
}

}  // namespace mla

using namespace mla;

extern "C" {

const char* mla_status_string(mla_status_t s) {
    switch (s) {
        case MLA_OK: return "MLA_OK";
        case MLA_ERR_INVALID_ARG: return "MLA_ERR_INVALID_ARG";
        case MLA_ERR_UNSUPPORTED: return "MLA_ERR_UNSUPPORTED";
        case MLA_ERR_CUDA: return "MLA_ERR_CUDA";
        case MLA_ERR_NO_MEMORY: return "MLA_ERR_NO_MEMORY";
        case MLA_ERR_DEVICE: return "MLA_ERR_DEVICE";
    }
    return "MLA_ERR_UNKNOWN";
}

const char* mla_last_error(void) { return t_last_error.c_str(); }

int32_t mla_set_impl(int32_t impl) { return g_impl.exchange(impl); }

int32_t mla_last_decode_impl(void) { return t_last_impl; }

constexpr int64_t kChunkCapPages = 160;  // 10,240 positions

int32_t mla_auto_splits(int32_t B, int32_t T, int32_t H, int32_t max_pages, int32_t sm_count) {
    if (B <= 0 || max_pages <= 2) return 1;
    // Units of more than 16 rows (t, h) run on the wide kernel: ceil(rows / 32)
    // CTAs per unit.
    const int64_t rows = (int64_t)(T > 0 ? T : 1) * (H > 0 ? H : 1);
    const int64_t G = rows > 16 ? ceil_div(rows, 32) : 1;
    if (sm_count <= 0) {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            cudaGetLastError();
            sm_count = 148;
        }
    }
    const int64_t most = ceil_div(max_pages, 2);
    // G CTAs per unit (1 for the 12-head kernel): the count that minimises waves
    // of CTAs x (pages per partition + a fixed cost of ~8 pages per CTA),
    // assuming every request is max_pages long.  A count that overshoots a wave
    // by a few units (e.g. ceil(SMs / B) partitions per request) pays a second wave.
    int64_t best = -1, s = 1;
    for (int64_t c = 1; c <= most && c <= 1024; ++c) {
        const int64_t cost = ceil_div(B * c * G, sm_count) * (ceil_div(max_pages, c) + 8);
        if (best < 0 || cost < best) best = cost, s = c;
    }
    // Partitions of at most kChunkCapPages pages: in a batch of mixed lengths the
    // longest request would otherwise bound the call (the host cannot see the
    // lengths); partitions past a request's end cost a CTA that exits at once.
    if (s < ceil_div(max_pages, kChunkCapPages)) s = ceil_div(max_pages, kChunkCapPages);
    if (s > most) s = most;
    if (s < 1) s = 1;
    // Snap to the count that equal chunks actually produce.
    const int64_t chunk = mla_split_chunk_pages(max_pages, (int32_t)s);
    return (int32_t)ceil_div(max_pages, chunk);
}

// Costs of the length-aware plan, in eighths of a page of loop time (~0.74 us
// per page under a full wave): a partition costs its pages plus a fixed 8
// pages per CTA (set-up ~3-4.5 us and epilogue ~2-2.4 us); a CTA whose
// partition lies past its request's history costs ~0.75 page in a
// longest-first launch, where it still starts after all the others.
constexpr int64_t kPlanPage = 8;
constexpr int64_t kPlanFixed = 8 * kPlanPage;
constexpr int64_t kPlanEmpty = 6;
// Both tensor-core kernels take the units of at most this many requests in
// longest-first order when their CTAs outnumber the SMs (the ordering
// kernel's limit).
constexpr int32_t kLongestFirstMaxBatch = 1024;

int32_t mla_plan_splits(int32_t B, int32_t T, int32_t H, const int32_t* host_seq_lens, int32_t max_pages,
                        int32_t sm_count) {
    const int32_t fallback = mla_auto_splits(B, T, H, max_pages, sm_count);
    if (!host_seq_lens || B <= 0 || max_pages <= 2) return fallback;
    const int64_t rows = (int64_t)(T > 0 ? T : 1) * (H > 0 ? H : 1);
    const bool narrow = rows <= 16;  // the 12-head kernel: one CTA per unit
    const int64_t G = narrow ? 1 : ceil_div(rows, 32);
    if (sm_count <= 0) {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            cudaGetLastError();
            sm_count = 148;
        }
    }
    std::vector<int64_t> pages(B);
    for (int32_t b = 0; b < B; ++b) {
        int64_t L = host_seq_lens[b];
        L = L < 0 ? 0 : (L > (int64_t)max_pages * kPage ? (int64_t)max_pages * kPage : L);
        pages[b] = ceil_div(L, kPage);
    }
    // Candidate counts: up to 8 waves of CTAs at full length (more never pays)
    // and, for the 12-head kernel, partitions down to 64 pages (a batch of
    // uneven lengths leaves most of its units empty); one per distinct chunk
    // size.  Each has a lower bound on its finish (its longest CTA, and its
    // total work spread over every SM); candidates are replayed in the order
    // of that bound until the bound passes the best finish found, which gives
    // the same answer as replaying them all.
    const int64_t most = ceil_div(max_pages, 2);
    int64_t hi = (8 * (int64_t)sm_count) / (B * G);
    if (narrow) hi = std::max<int64_t>(hi, ceil_div(max_pages, 64));
    hi = hi < 1 ? 1 : (hi > most ? most : hi);
    if (hi > 1024) hi = 1024;
    const int64_t longest = *std::max_element(pages.begin(), pages.end());
    struct Cand {
        int64_t bound, n, chunk;
    };
    std::vector<Cand> cands;
    for (int64_t c = 1, last_chunk = -1; c <= hi; ++c) {
        const int64_t chunk = mla_split_chunk_pages(max_pages, (int32_t)c);
        if (chunk == last_chunk) continue;  // the same snapped plan as a smaller count
        last_chunk = chunk;
        int64_t work = 0;
        for (int64_t p : pages) work += kPlanPage * p + ceil_div(p, chunk) * kPlanFixed;
        const int64_t bound =
            std::max(kPlanPage * std::min(chunk, longest) + kPlanFixed, ceil_div(G * work, sm_count));
        cands.push_back({bound, ceil_div(max_pages, chunk), chunk});
    }
    std::sort(cands.begin(), cands.end(),
              [](const Cand& a, const Cand& b) { return a.bound != b.bound ? a.bound < b.bound : a.n < b.n; });
    std::vector<int64_t> load((size_t)sm_count), partial;
    int64_t best_cost = -1, best = 1;
    for (const Cand& cd : cands) {
        if (best_cost >= 0 && (cd.bound > best_cost || (cd.bound == best_cost && cd.n > best))) break;
        // Each CTA starts on the SM that frees first, one CTA per SM.
        std::fill(load.begin(), load.end(), 0);  // all zero: already a heap
        int64_t cost = 0;                         // the latest finish so far
        auto place = [&](int64_t w) {
            std::pop_heap(load.begin(), load.end(), std::greater<int64_t>());
            load.back() += w;
            cost = std::max(cost, load.back());
            std::push_heap(load.begin(), load.end(), std::greater<int64_t>());
        };
        const bool longest_first =
            cd.n > 1 && B <= kLongestFirstMaxBatch && (int64_t)B * cd.n * G > sm_count;
        if (longest_first) {
            // full chunks request by request, then the partial chunks by length,
            // then the CTAs of the partitions past each history; a unit's G
            // row-CTAs start one after another
            int64_t live = 0;
            partial.clear();
            for (int32_t b = 0; b < B; ++b) {
                const int64_t f = pages[b] / cd.chunk, r = pages[b] - f * cd.chunk;
                for (int64_t i = 0; i < f * G; ++i) place(kPlanPage * cd.chunk + kPlanFixed);
                live += f;
                if (r > 0) partial.push_back(r);
            }
            std::sort(partial.begin(), partial.end(), std::greater<int64_t>());
            for (int64_t r : partial)
                for (int64_t i = 0; i < G; ++i) place(kPlanPage * r + kPlanFixed);
            live += (int64_t)partial.size();
            for (int64_t e = live * G; e < (int64_t)B * cd.n * G; ++e) place(kPlanEmpty);
        } else {
            // launch order: partition and row-CTA fastest, then the request
            for (int32_t b = 0; b < B; ++b) {
                for (int64_t sp = 0; sp < cd.n; ++sp) {
                    const int64_t w = std::min(cd.chunk, pages[b] - sp * cd.chunk);
                    if (w <= 0) break;  // partitions past the request's end exit at once
                    for (int64_t r = 0; r < G; ++r) place(kPlanPage * w + kPlanFixed);
                }
            }
        }
        if (best_cost < 0 || cost < best_cost || (cost == best_cost && cd.n < best)) best_cost = cost, best = cd.n;
    }
    return (int32_t)best;
}

int32_t mla_split_chunk_pages(int32_t max_pages, int32_t n_splits) {
    if (max_pages <= 0) return 1;
    if (n_splits < 1) n_splits = 1;
    const int64_t chunk = ceil_div(max_pages, n_splits);
    return (int32_t)(chunk < 1 ? 1 : chunk);
}

size_t mla_decode_workspace_bytes(int32_t B, int32_t T, int32_t H, int32_t n_splits) {
    if (n_splits <= 1 || B <= 0) return 0;
    const size_t rows = (size_t)B * T * H;
    const size_t out_bytes = (size_t)n_splits * rows * kDv * sizeof(float);
    const size_t lse_bytes = (size_t)n_splits * rows * sizeof(float);
    const size_t order_bytes = (size_t)n_splits * B * 2 * sizeof(int32_t);  // longest-first unit order
    return ((out_bytes + 255) & ~size_t(255)) + ((lse_bytes + 255) & ~size_t(255)) + order_bytes;
}

mla_status_t mla_device_error(int32_t* code, void* stream) {
    if (!code) return fail(MLA_ERR_INVALID_ARG, "code: null pointer");
    DeviceInfo* d = nullptr;
    mla_status_t st = device_info(&d);
    if (st != MLA_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    int v = 0;
    e = cudaMemcpy(&v, d->err_word, sizeof v, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpy(device error word)");
    if (v != 0) {
        const int zero = 0;
        e = cudaMemcpy(d->err_word, &zero, sizeof zero, cudaMemcpyHostToDevice);
        if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpy(clear device error word)");
    }
    *code = v;
    return MLA_OK;
}

mla_status_t mla_decode_paged(const mla_tensor_t* q, const mla_tensor_t* kv_cache,
                              const float* kv_scale, const mla_tensor_t* block_table,
                              const mla_tensor_t* seq_lens, int32_t n_splits, float sm_scale,
                              const mla_tensor_t* out, const mla_tensor_t* lse, void* stream) {
    t_last_error.clear();
    DecodeParams p{};
    bool empty = false;
    mla_status_t st = internal_prepare_decode(q, kv_cache, kv_scale, block_table, seq_lens, n_splits, 0,
                                              sm_scale, out, lse, &p, &empty);
    if (st != MLA_OK || empty) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (p.n_splits > 1) {
        void* ws = nullptr;
        const size_t need = mla_decode_workspace_bytes(p.B, p.T, p.H, p.n_splits);
        if ((st = get_scratch(need, s, &ws)) != MLA_OK) return st;
        internal_carve_scratch(p, ws);
    }
    return internal_launch_decode(p, s);
}

mla_status_t mla_profile_next_decode(void* ev_begin, void* ev_end) {
    t_prof_begin = static_cast<cudaEvent_t>(ev_begin);
    t_prof_end = static_cast<cudaEvent_t>(ev_end);
    return MLA_OK;
}

mla_status_t mla_release_graph_scratch(void) {
    t_last_error.clear();
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    std::lock_guard<std::mutex> lk(g_ws_mu);
    // the current device's retired buffers, and the live buffers that a
    // capture used (the next call on their stream allocates anew)
    std::vector<void*> drop;
    for (auto it = g_ws_retired.begin(); it != g_ws_retired.end();) {
        if (it->first == dev) {
            drop.push_back(it->second);
            it = g_ws_retired.erase(it);
        } else {
            ++it;
        }
    }
    for (auto& kv : g_ws) {
        if (kv.first.first == dev && kv.second.in_graph && kv.second.ptr) {
            drop.push_back(kv.second.ptr);
            kv.second = Scratch{};
        }
    }
    if (drop.empty()) return MLA_OK;
    // cudaFree waits for the device; a buffer freed here is in no stream's use
    for (void* ptr : drop) {
        e = cudaFree(ptr);
        if (e != cudaSuccess) return cuda_fail(e, "cudaFree(graph scratch)");
    }
    return MLA_OK;
}

int mla_test_stall_copies(int on) {
    const int prev = t_test_stall;
    t_test_stall = on ? 1 : 0;
    return prev;
}

int mla_test_count_rescales(int32_t* device_counts) {
    t_test_counts = device_counts;
    return MLA_OK;
}

mla_status_t mla_merge_partials(const mla_tensor_t* partial_out, const mla_tensor_t* partial_lse,
                                int32_t n_shards, const mla_tensor_t* out, const mla_tensor_t* lse,
                                void* stream) {
    t_last_error.clear();
    if (!partial_out || !partial_lse || !out)
        return fail(MLA_ERR_INVALID_ARG, "partial_out, partial_lse and out are required");
    const int nd = partial_out->ndim;
    if (nd < 2 || nd > 5) return fail(MLA_ERR_INVALID_ARG, "partial_out: rank must be 2..5");
    const int dt = partial_out->dtype;
    if (dt != MLA_DTYPE_BF16 && dt != MLA_DTYPE_F32)
        return fail(MLA_ERR_INVALID_ARG, "partial_out: dtype must be bf16 or fp32");
    mla_status_t st;
    if ((st = check_tensor(partial_out, "partial_out", nd, dt, true, 16)) != MLA_OK) return st;
    if (partial_out->shape[nd - 1] != kDv) return fail(MLA_ERR_UNSUPPORTED, "partial_out: last dim must be 512");
    if (n_shards < 1 || n_shards > 4096 || partial_out->shape[0] != n_shards)
        return fail(MLA_ERR_INVALID_ARG, "n_shards must equal partial_out.shape[0] and lie in [1, 4096]");
    if ((st = check_tensor(partial_lse, "partial_lse", nd - 1, MLA_DTYPE_F32, true, 4)) != MLA_OK) return st;
    int64_t rows = 1;
    for (int i = 0; i < nd - 1; ++i)
        if (partial_lse->shape[i] != partial_out->shape[i])
            return fail(MLA_ERR_INVALID_ARG, "partial_lse: shape must be partial_out.shape[:-1]");
    for (int i = 1; i < nd - 1; ++i) rows *= partial_out->shape[i];
    if ((st = check_tensor(out, "out", nd - 1, MLA_DTYPE_BF16, true, 16)) != MLA_OK) return st;
    for (int i = 1; i < nd; ++i)
        if (out->shape[i - 1] != partial_out->shape[i])
            return fail(MLA_ERR_INVALID_ARG, "out: shape must be partial_out.shape[1:]");
    if (lse) {
        if (nd - 2 == 0) return fail(MLA_ERR_INVALID_ARG, "lse: rank-0 output not supported; pass NULL");
        if ((st = check_tensor(lse, "lse", nd - 2, MLA_DTYPE_F32, true, 4)) != MLA_OK) return st;
        for (int i = 1; i < nd - 1; ++i)
            if (lse->shape[i - 1] != partial_out->shape[i])
                return fail(MLA_ERR_INVALID_ARG, "lse: shape must be partial_out.shape[1:-1]");
    }
    if (rows == 0) return MLA_OK;
    MergeParams m{};
    m.part_out = partial_out->data;
    m.part_lse = static_cast<const float*>(partial_lse->data);
    m.S = n_shards;
    m.rows = rows;
    m.in_bf16 = dt == MLA_DTYPE_BF16;
    m.out = static_cast<uint16_t*>(out->data);
    m.lse = lse ? static_cast<float*>(lse->data) : nullptr;
    m.pdl = 0;
    cudaError_t e = launch_merge(m, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "merge launch");
    return MLA_OK;
}

}  // extern "C"

int mla_bench_stream_pages(const void* kv_cache, int64_t num_pages, const int32_t* page_ids, int32_t ctas,
                           int32_t pages_per_cta, void* stream) {
    using namespace mla;
    if (!kv_cache || !page_ids) return fail(MLA_ERR_INVALID_ARG, "mla_bench_stream_pages: null pointer");
    if ((reinterpret_cast<uintptr_t>(kv_cache) & 15) != 0)
        return fail(MLA_ERR_INVALID_ARG, "mla_bench_stream_pages: kv_cache must be 16-byte aligned");
    if (num_pages < 1 || num_pages * kPage >= (int64_t(1) << 31))
        return fail(MLA_ERR_INVALID_ARG, "mla_bench_stream_pages: num_pages out of range");
    if (ctas < 1 || ctas > 65535 || pages_per_cta < 1)
        return fail(MLA_ERR_INVALID_ARG, "mla_bench_stream_pages: ctas in [1, 65535], pages_per_cta >= 1");
    DeviceInfo* dev = nullptr;
    mla_status_t st = device_info(&dev);
    if (st != MLA_OK) return st;
    cudaError_t e = launch_stream_probe(static_cast<const uint8_t*>(kv_cache), num_pages, page_ids, ctas,
                                        pages_per_cta, dev->err_word, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "stream probe launch");
    return MLA_OK;
}
