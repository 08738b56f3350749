"""Host-side checks of the C ABI (no GPU needed): the library loads, exports
every symbol the header declares, plans splits as documented and rejects bad
arguments before touching the device."""
import ctypes
import os
import re

import numpy as np
import pytest
import torch

from mla_latent_kv_fp8_gb300 import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    from mla_latent_kv_fp8_gb300 import build
    build.build()
    from mla_latent_kv_fp8_gb300 import _lib
    return _lib


def _declared_functions():
    names = []
    inc = os.path.join(ROOT, "include")
    for f in sorted(os.listdir(inc)):
        if f.endswith(".h"):
            src = open(os.path.join(inc, f)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names += re.findall(r"\b(mla_[a-z_0-9]+)\s*\(", src)
    return sorted(set(names))


def test_library_exports_every_declared_symbol(L):
    lib = L.lib()
    declared = _declared_functions()
    assert "mla_decode_paged" in declared and "mla_merge_partials" in declared
    for name in declared:
        assert hasattr(lib, name), f"{name} declared in include/ but not exported"
    assert set(L.EXPORTS) <= set(declared)


def test_status_strings(L):
    assert L.mla_status_string(0) == "MLA_OK"
    assert L.mla_status_string(2) == "MLA_ERR_UNSUPPORTED"
    assert L.mla_status_string(99) == "MLA_ERR_UNKNOWN"


@pytest.mark.parametrize("B,max_pages,sm,expect", [
    (8, 512, 152, 19),      # 8 requests x 32K: one wave of 152 units
    (1, 6144, 152, 150),    # one request x 393K: >= SM count partitions
    (1, 16, 152, 8),        # short history: partitions of >= 2 pages
    (1, 2, 152, 1),
    (200, 100, 152, 3),     # more requests than SMs: 4 waves of 34-page partitions beat 2 unsplit
    (16, 512, 152, 9),      # 144 units in one wave (ceil(152 / 16) = 10 would spill 8 into a second)
    (32, 512, 152, 9),      # 288 units: two nearly full waves of 57 pages
    (128, 2219, 152, 14),   # the ragged mix's table: 160-page partitions
])
def test_auto_splits(L, B, max_pages, sm, expect):
    s = L.mla_auto_splits(B, 1, 12, max_pages, sm)
    assert s == expect
    chunk = L.mla_split_chunk_pages(max_pages, s)
    assert chunk >= 1
    assert -(-max_pages // chunk) == s  # every partition non-empty at full length


@pytest.mark.parametrize("B,T,H,max_pages,sm,expect", [
    (32, 1, 96, 278, 152, 3),      # 96 rows: 3 wide CTAs per unit, wave cost model (288 CTAs)
    (16, 4, 12, 1568, 152, 14),    # 48 rows: 2 wide CTAs per unit, wave cost model (448 CTAs)
    (128, 1, 12, 2219, 152, 14),   # many requests of mixed length: the 160-page cap
    (8, 1, 12, 512, 152, 19),      # one wave, as before
])
def test_auto_splits_rows_and_cap(L, B, T, H, max_pages, sm, expect):
    s = L.mla_auto_splits(B, T, H, max_pages, sm)
    assert s == expect
    chunk = L.mla_split_chunk_pages(max_pages, s)
    assert chunk <= 160
    assert -(-max_pages // chunk) == s


def test_workspace_bytes(L):
    assert L.mla_decode_workspace_bytes(8, 1, 12, 1) == 0
    n = L.mla_decode_workspace_bytes(8, 1, 12, 19)
    assert n >= 19 * 8 * 12 * 513 * 4


def _desc(shape, dtype_code, ptr=0x10000):
    d = L_mod().mla_tensor_t()
    d.data = ptr
    st = 1
    strides = []
    for s in reversed(shape):
        strides.append(st)
        st *= s
    strides.reverse()
    for i, (s, k) in enumerate(zip(shape, strides)):
        d.shape[i] = s
        d.stride[i] = k
    d.ndim = len(shape)
    d.dtype = dtype_code
    return d


def L_mod():
    from mla_latent_kv_fp8_gb300 import _lib
    return _lib


def _call_decode(L, q, kv, bt, sl, out, lse, n_splits=0, scale_ptr=0x20000):
    lib = L.lib()
    ref = lambda d: ctypes.byref(d) if d is not None else None  # noqa: E731
    return lib.mla_decode_paged(ref(q), ref(kv), ctypes.c_void_p(scale_ptr), ref(bt), ref(sl),
                                n_splits, 0.07, ref(out), ref(lse), None)


def _good(B=2, T=1, H=12, mp=4, npages=8):
    return dict(q=_desc([B, T, H, 576], 1), kv=_desc([npages, 64, 576], 3), bt=_desc([B, mp], 4),
                sl=_desc([B], 4), out=_desc([B, T, H, 512], 1), lse=_desc([B, T, H], 2))


@pytest.mark.parametrize("mutate,status", [
    (lambda a: a.update(q=None), 1),
    (lambda a: setattr(a["q"], "dtype", 2), 1),
    (lambda a: a.update(q=_desc([2, 1, 12, 512], 1)), 2),      # dims other than 576
    (lambda a: a.update(q=_desc([2, 2, 96, 576], 1),
                        out=_desc([2, 2, 96, 512], 1), lse=_desc([2, 2, 96], 2)), 2),  # H*T > 128
    (lambda a: a.update(kv=_desc([8, 32, 576], 3)), 2),         # page size 32
    (lambda a: a.update(bt=_desc([3, 4], 4)), 1),
    (lambda a: a.update(sl=_desc([2], 2)), 1),
    (lambda a: a.update(out=_desc([2, 1, 12, 576], 1)), 1),
    (lambda a: a.update(lse=_desc([2, 1, 11], 2)), 1),
    (lambda a: setattr(a["q"], "data", 0x10008), 2),           # misaligned q
    (lambda a: a["q"].stride.__setitem__(3, 2), 2),            # non-contiguous q
])
def test_decode_rejects_bad_arguments_on_host(L, mutate, status):
    a = _good()
    mutate(a)
    st = _call_decode(L, a["q"], a["kv"], a["bt"], a["sl"], a["out"], a["lse"])
    assert st == status, L.mla_last_error()
    assert L.mla_last_error() != ""


def test_decode_rejects_negative_splits_and_null_scale(L):
    a = _good()
    assert _call_decode(L, a["q"], a["kv"], a["bt"], a["sl"], a["out"], a["lse"], n_splits=-1) == 1
    assert _call_decode(L, a["q"], a["kv"], a["bt"], a["sl"], a["out"], a["lse"], scale_ptr=0) == 1


def test_empty_batch_is_a_no_op(L):
    a = _good(B=0)
    assert _call_decode(L, a["q"], a["kv"], a["bt"], a["sl"], a["out"], a["lse"]) == 0


def test_merge_rejects_bad_arguments_on_host(L):
    lib = L.lib()
    po, pl = _desc([4, 3, 512], 2), _desc([4, 3], 2)
    out, lse = _desc([3, 512], 1), _desc([3], 2)
    r = ctypes.byref
    assert lib.mla_merge_partials(r(po), r(pl), 5, r(out), r(lse), None) == 1      # n_shards mismatch
    assert lib.mla_merge_partials(r(po), r(_desc([4, 2], 2)), 4, r(out), r(lse), None) == 1
    assert lib.mla_merge_partials(r(_desc([4, 3, 256], 2)), r(pl), 4, r(_desc([3, 256], 1)),
                                  r(lse), None) == 2
    assert lib.mla_merge_partials(r(_desc([4, 3, 512], 4)), r(pl), 4, r(out), r(lse), None) == 1
    assert lib.mla_merge_partials(r(po), r(pl), 4, r(_desc([3, 512], 2)), r(lse), None) == 1


def test_binding_maps_torch_dtypes(L):
    d = L.describe(torch.zeros(2, 3, dtype=torch.bfloat16))
    assert d.ndim == 2 and d.dtype == 1 and d.shape[1] == 3 and d.stride[0] == 3
    assert L.describe(torch.zeros(1, dtype=torch.float8_e4m3fn)).dtype == 3
    assert L.describe(torch.zeros(1, dtype=torch.int32)).dtype == 4
    assert L.describe(None) is None


def test_stream_probe_rejects_bad_arguments_on_host(L):
    lib = L.lib()
    ids = ctypes.c_void_p(4096)  # never dereferenced: every case fails validation first
    assert lib.mla_bench_stream_pages(None, 8, ids, 1, 1, None) == 1
    assert lib.mla_bench_stream_pages(ctypes.c_void_p(4096), 8, None, 1, 1, None) == 1
    assert lib.mla_bench_stream_pages(ctypes.c_void_p(4100), 8, ids, 1, 1, None) == 1   # not 16-byte aligned
    assert lib.mla_bench_stream_pages(ctypes.c_void_p(4096), 0, ids, 1, 1, None) == 1   # no pages
    assert lib.mla_bench_stream_pages(ctypes.c_void_p(4096), 1 << 25, ids, 1, 1, None) == 1
    assert lib.mla_bench_stream_pages(ctypes.c_void_p(4096), 8, ids, 0, 1, None) == 1   # no CTAs
    assert lib.mla_bench_stream_pages(ctypes.c_void_p(4096), 8, ids, 1, 0, None) == 1


def _call_append(L, lat, bt, sp, kv, scale_ptr=0x20000):
    ref = lambda d: ctypes.byref(d) if d is not None else None  # noqa: E731
    return L.lib().mla_append_latent(ref(lat), ctypes.c_void_p(scale_ptr), ref(bt), ref(sp), ref(kv), None)


def _good_append(B=2, T=1, mp=4, npages=8):
    return dict(lat=_desc([B, T, 576], 1), bt=_desc([B, mp], 4), sp=_desc([B], 4), kv=_desc([npages, 64, 576], 3))


@pytest.mark.parametrize("mutate,status", [
    (lambda a: a.update(lat=None), 1),
    (lambda a: setattr(a["lat"], "dtype", 2), 1),                 # fp32 latents
    (lambda a: a.update(lat=_desc([2, 1, 512], 1)), 2),           # 512-wide latents
    (lambda a: a.update(bt=_desc([3, 4], 4)), 1),                 # block table of 3 requests
    (lambda a: a.update(sp=_desc([3], 4)), 1),                    # start positions of 3 requests
    (lambda a: a.update(sp=_desc([2], 2)), 1),                    # fp32 start positions
    (lambda a: a.update(kv=_desc([8, 32, 576], 3)), 2),           # page size 32
    (lambda a: a.update(kv=_desc([8, 64, 576], 1)), 1),           # bf16 cache
    (lambda a: setattr(a["lat"], "data", 0x10008), 2),           # misaligned latents
    (lambda a: a["kv"].stride.__setitem__(1, 1152), 2),          # non-contiguous cache
])
def test_append_rejects_bad_arguments_on_host(L, mutate, status):
    a = _good_append()
    mutate(a)
    st = _call_append(L, a["lat"], a["bt"], a["sp"], a["kv"])
    assert st == status, L.mla_last_error()
    assert L.mla_last_error() != ""


def test_append_null_scale_and_empty_batch(L):
    a = _good_append()
    assert _call_append(L, a["lat"], a["bt"], a["sp"], a["kv"], scale_ptr=0) == 1
    a = _good_append(B=0)
    assert _call_append(L, a["lat"], a["bt"], a["sp"], a["kv"]) == 0
    a = _good_append(T=0)
    assert _call_append(L, a["lat"], a["bt"], a["sp"], a["kv"]) == 0


def test_auto_splits_invariants_over_a_sweep(L):
    """Over a sweep of batch shapes: the plan is snapped to equal chunks that all
    start inside the table, no chunk exceeds 160 pages or falls below 2, and a
    long enough batch of units of at most 16 rows fills most of a wave of SMs."""
    for B in (1, 2, 3, 8, 16, 31, 64, 128, 1000):
        for T, H in ((1, 12), (1, 16), (4, 12), (1, 96), (2, 64), (1, 128)):
            for max_pages in (1, 2, 3, 5, 16, 64, 100, 161, 512, 2219, 6144, 40000):
                for sm in (148, 152):
                    s = L.mla_auto_splits(B, T, H, max_pages, sm)
                    chunk = L.mla_split_chunk_pages(max_pages, s)
                    assert s >= 1 and chunk >= 1
                    assert -(-max_pages // chunk) == s
                    assert chunk <= 160 or s == 1 and max_pages <= 2
                    if max_pages > 2:
                        assert chunk >= 2
                    if T * H <= 16 and max_pages >= 2 * sm:
                        # enough pages: the (request, partition) units fill most of
                        # a wave (equal chunks of whole pages can drop a few)
                        assert B * s >= 0.8 * sm


@pytest.mark.parametrize("B,T,H,max_pages", [
    (32, 1, 96, 278),    # dcp_shard
    (16, 4, 12, 1568),   # verify-like, 48 rows
    (16, 1, 48, 195),    # a DCP-verify shard before the last
    (3, 2, 64, 700),     # 128 rows, 4 CTAs per unit
    (8, 1, 12, 512),     # tp8_batch: one wave of 12-head units
    (1, 1, 12, 6144),    # the 393,216-position request
])
def test_plan_splits_equals_auto_when_every_request_is_full(L, B, T, H, max_pages):
    """With every request max_pages long the length-aware plan and the automatic
    one agree (both minimise waves x partition length for uniform work)."""
    full = [64 * max_pages] * B
    assert L.mla_plan_splits(B, T, H, full, max_pages, 152) == L.mla_auto_splits(B, T, H, max_pages, 152)


def test_plan_splits_falls_back_to_auto(L):
    """Without host lengths (or requests) the plan is the automatic count."""
    lens = [1000, 20000, 5, 0, 70000, 3000, 64, 9000]
    mp = -(-max(lens) // 64)
    for T, H in ((1, 12), (1, 16), (2, 8), (4, 12)):
        assert L.lib().mla_plan_splits(8, T, H, None, mp, 152) == L.mla_auto_splits(8, T, H, mp, 152)
        assert L.mla_plan_splits(0, T, H, [], mp, 152) == L.mla_auto_splits(0, T, H, mp, 152)


def test_plan_splits_for_uneven_12_head_batches(L):
    """12-head units: one wave while the units fit the SMs, and past that the
    longest-first launch.  An uneven batch of 8 takes short partitions so that
    its longest request spreads over the SMs its short ones leave free; the
    seeded 128-request ragged mix takes 5 partitions: the fastest count of a
    sweep on GB300 (342.2 us per step, against 343.7 at 10, 349.5 at 15,
    357.3 at the automatic 14, 369.5 at 4, 385.0 at 8)."""
    lens = [1000, 20000, 5, 0, 70000, 3000, 64, 9000]
    mp = -(-max(lens) // 64)
    n = L.mla_plan_splits(8, 1, 12, lens, mp, 152)
    assert n > L.mla_auto_splits(8, 1, 12, mp, 152)
    chunk = L.mla_split_chunk_pages(mp, n)
    assert sum(-(-(-(-x // 64)) // chunk) for x in lens) <= 152  # still one wave
    ragged = synth.ragged_lens(6)
    mp = -(-max(ragged) // 64)
    assert L.mla_plan_splits(128, 1, 12, ragged, mp, 152) == 5
    assert L.mla_auto_splits(128, 1, 12, mp, 152) == 14


def test_plan_splits_ragged_batches(L):
    """Uneven histories on the 32-row kernel: the plan replays the
    longest-first launch its CTA count triggers.  On the verify workload's 8-way
    DCP shards (16 requests x 48 rows, 16..195 pages) and on the whole verify
    workload it picks 8 partitions (measured on GB300: the shard rank step
    41.5 us against 43.9 us at the 7 a request-order plan took; the whole
    workload 160.4 us per step against 173.9 us at 16 in request order, 172.4 us
    at 16 and 215.7 us at 8 in request order)."""
    from mla_latent_kv_fp8_gb300.dcp import shard_plan
    lens = synth.verify_lens(4)
    Lb = L
    plan = shard_plan(lens, torch.zeros((16, 2048), dtype=torch.int32), 8, 4)
    for (table, sl), (T, H) in ((plan[0], (1, 48)), (plan[-1], (4, 12))):
        assert Lb.mla_plan_splits(16, T, H, sl.tolist(), table.shape[1], 152) == 8
    mp = -(-max(lens) // 64)
    assert Lb.mla_plan_splits(16, 4, 12, lens, mp, 152) == 8
    assert Lb.mla_auto_splits(16, 4, 12, mp, 152) == 14


def test_plan_splits_is_a_valid_plan_over_a_sweep(L):
    rng = np.random.default_rng(5)
    for _ in range(200):
        B = int(rng.integers(1, 40))
        T = int(rng.choice([1, 2, 4, 8]))
        H = int(rng.integers(1, 128 // T + 1))
        lens = [int(x) for x in rng.integers(-5, 200_000, size=B)]
        mp = max(1, -(-max(max(lens), 0) // 64) + int(rng.integers(0, 3)))
        n = L.mla_plan_splits(B, T, H, lens, mp, int(rng.choice([148, 152])))
        chunk = L.mla_split_chunk_pages(mp, n)
        assert 1 <= n and -(-mp // chunk) == n
        if mp > 2:
            assert n <= -(-mp // 2)


def _plan_by_replay(B, T, H, lens, max_pages, sm):
    """The length-aware plan written out plainly: every candidate count (one per
    distinct chunk size, up to 8 full-length waves, and for units of at most
    16 rows partitions down to 64 pages) replayed on a min-heap of SM finish
    times, in eighths of a page: a partition costs 8 per page plus 64 on each of
    its row-CTAs, in launch order; a launch of more CTAs than SMs (at most 1,024
    requests) runs full chunks first, then partial chunks longest first, then
    the partitions past each history at 6 per CTA.  The earliest finish wins,
    ties to fewer partitions."""
    import heapq
    narrow = T * H <= 16
    G = 1 if narrow else -(-(T * H) // 32)
    pages = [-(-min(max(x, 0), 64 * max_pages) // 64) for x in lens]
    most = -(-max_pages // 2)
    hi = (8 * sm) // (B * G)
    if narrow:
        hi = max(hi, -(-max_pages // 64))
    hi = max(1, min(most, hi, 1024))
    best = None
    seen = set()
    for c in range(1, hi + 1):
        chunk = max(1, -(-max_pages // c))
        if chunk in seen:
            continue
        seen.add(chunk)
        n = -(-max_pages // chunk)
        heap = [0] * sm
        finish = 0

        def place(w):
            nonlocal finish
            t = heapq.heappop(heap) + w
            finish = max(finish, t)
            heapq.heappush(heap, t)

        if n > 1 and B <= 1024 and B * n * G > sm:
            full = [chunk] * sum(p // chunk for p in pages)
            part = sorted((p % chunk for p in pages if p % chunk), reverse=True)
            for w in full + part:
                for _ in range(G):
                    place(8 * w + 64)
            for _ in range((B * n - len(full) - len(part)) * G):
                place(6)
        else:
            for p in pages:
                for s in range(n):
                    w = min(chunk, p - s * chunk)
                    if w <= 0:
                        break
                    for _ in range(G):
                        place(8 * w + 64)
        if best is None or (finish, n) < best:
            best = (finish, n)
    return best[1]


def test_plan_splits_matches_a_plain_replay(L):
    """The library's pruned search returns what replaying every candidate returns,
    for the 32-row kernel and for 12-head units (one wave and longest-first)."""
    rng = np.random.default_rng(11)
    for i in range(90):
        T = int(rng.choice([1, 2, 4]))
        if i % 3 == 2:  # at most 16 rows, batches up to past the longest-first limit
            B = int(rng.choice([int(rng.integers(1, 40)), int(rng.integers(100, 300)), 1030]))
            H = int(rng.integers(1, 16 // T + 1))
        else:
            B = int(rng.integers(1, 40))
            H = int(rng.integers(17 // T + 1, 128 // T + 1))  # more than 16 rows
        lens = [int(x) for x in rng.integers(0, int(rng.choice([3000, 40000, 150000])), size=B)]
        mp = max(3, -(-max(lens) // 64))
        sm = int(rng.choice([148, 152]))
        assert L.mla_plan_splits(B, T, H, lens, mp, sm) == _plan_by_replay(B, T, H, lens, mp, sm), (B, T, H, mp)
