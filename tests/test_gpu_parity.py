"""GPU parity: the CUDA path (through the C ABI) against the FP64 oracle on the
same seeded bytes, element by element, within the stated tolerances.

Reduced-size cases compare every output; full-size workloads (the shapes the
benchmark times, in the same launch configuration) compare sampled rows that
the oracle computes one by one.  Output buffers are filled with NaN first so
that an unwritten element fails."""
import math

import numpy as np
import pytest
import torch

import oracle
from mla_latent_kv_fp8_gb300 import synth
from tests.parity import assert_parity

pytestmark = pytest.mark.gpu

IMPLS = {"simt": 1, "tcgen05": 2}


@pytest.fixture(scope="module")
def L():
    from mla_latent_kv_fp8_gb300 import build
    build.build()
    from mla_latent_kv_fp8_gb300 import _lib
    _lib.lib()
    return _lib


@pytest.fixture(params=sorted(IMPLS))
def impl(request, L):
    prev = L.mla_set_impl(IMPLS[request.param])
    yield request.param
    L.mla_set_impl(prev)


def run(L, case, n_splits=0, with_lse=True, stream=None):
    B, T, H = case.q.shape[:3]
    out = torch.full((B, T, H, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((B, T, H), float("nan"), dtype=torch.float32, device="cuda") if with_lse else None
    L.mla_decode_paged(case.q, case.kv_cache, case.kv_scale, case.block_table, case.seq_lens,
                       n_splits, case.sm_scale, out, lse, stream)
    torch.cuda.synchronize()
    assert L.mla_device_error() == 0
    return out, lse


def supported(L, impl, case, n_splits=0):
    """The tensor-core family declines shapes it does not cover; that is an error only
    when it is the selected family."""
    try:
        return run(L, case, n_splits)
    except L.MlaError as e:
        if impl == "tcgen05" and e.status == 2:
            pytest.skip(f"tcgen05 kernel does not cover this shape: {e}")
        raise


def oracle_full(case):
    c = case.to("cpu")
    return oracle.decode(c.q, c.kv_cache, c.kv_scale, c.block_table, c.seq_lens, c.sm_scale)


def oracle_rows(case, reqs, heads):
    """Oracle for the sampled requests/heads, on a compact identity-paged copy of
    just those requests' pages (paging invariance is pinned separately)."""
    reqs = list(reqs)
    lens = [case.lens[b] for b in reqs]
    pages = [(x + 63) // 64 for x in lens]
    bt = case.block_table[reqs].cpu().numpy()
    ids = np.concatenate([bt[i, :pages[i]] for i in range(len(reqs))]).astype(np.int64)
    kv = case.kv_cache[torch.from_numpy(ids).to(case.kv_cache.device)].cpu()
    bt_id = np.zeros((len(reqs), max(max(pages), 1)), dtype=np.int32)
    off = 0
    for i, p in enumerate(pages):
        bt_id[i, :p] = np.arange(off, off + p)
        off += p
    q = case.q[reqs].cpu()
    rm = np.zeros((len(reqs), case.T, case.H), dtype=np.uint8)
    rm[:, :, heads] = 1
    o, l = oracle.decode(q, kv, case.kv_scale.cpu(), torch.from_numpy(bt_id),
                         torch.tensor(lens, dtype=torch.int32), case.sm_scale, row_mask=rm)
    return o[:, :, heads], l[:, :, heads]


# ----------------------------------------------------------------------------
# Reduced sizes: every output against the oracle
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("name,n_splits", [
    ("tiny", 4), ("tiny", 1), ("tp8_batch", 0), ("tp8_batch", 1), ("tp8_batch", 3),
    ("tp8_batch", 7), ("verify", 0), ("verify", 5), ("long", 0), ("long", 200),
    ("ragged", 0), ("ragged", 9), ("dcp_shard", 0), ("dcp_shard", 2)])
def test_reduced_workloads_match_oracle(L, impl, name, n_splits):
    case = synth.workload_case(name, reduced=True)
    out, lse = supported(L, impl, case.to("cuda"), n_splits)
    ro, rl = oracle_full(case)
    assert_parity(out, lse, ro, rl, what=f"{name}/{impl}/splits={n_splits}")


@pytest.mark.parametrize("lens,H,T", [
    ([1], 12, 1), ([64], 12, 1), ([65], 12, 1), ([128, 129, 127], 12, 1), ([4, 5, 68], 12, 4),
    ([0, 300, 0], 12, 1), ([200], 1, 1), ([333, 17], 7, 3), ([260], 128, 1), ([190, 66], 32, 4),
    ([517], 16, 8), ([1000], 96, 1), ([300, 77], 14, 1), ([260, 9], 4, 4), ([700], 16, 1),
    # the wide kernel at its boundaries: 17 rows (1 CTA), 33 (2 CTAs of 17 + 16),
    # 65 (3 CTAs), 100 and 120 (4 CTAs), causal with 6 and 13 draft positions
    ([70, 1, 0], 17, 1), ([200, 129], 33, 1), ([640, 64], 5, 13), ([129], 100, 1), ([300], 20, 6)])
def test_edge_shapes_match_oracle(L, impl, lens, H, T):
    case = synth.make_decode_case(1000 + sum(lens) + H + T, lens, H, T, extra_pages=3)
    for n_splits in (0, 1, 3):
        out, lse = supported(L, impl, case.to("cuda"), n_splits)
        ro, rl = oracle_full(case)
        assert_parity(out, lse, ro, rl, what=f"lens={lens} H={H} T={T} splits={n_splits}")


def test_more_splits_than_pages(L, impl):
    case = synth.make_decode_case(77, [130, 5, 0], 12, 1)
    out, lse = supported(L, impl, case.to("cuda"), 64)
    ro, rl = oracle_full(case)
    assert_parity(out, lse, ro, rl, what="64 splits over <= 3 pages")


def test_unread_cache_bytes_do_not_leak(L, impl):
    """NaN codes (0x7F) beyond seq_len inside the last page and in pages no request
    references must not reach the output: only visible positions are read."""
    lens = [70, 200, 1]
    case = synth.make_decode_case(55, lens, 12, 1, extra_pages=4)
    kv = case.kv_cache.clone()
    bt = case.block_table.numpy()
    for b, L_ in enumerate(lens):
        last = (L_ - 1) // 64
        kv[bt[b, last], L_ % 64 or 64:, :] = 0x7F
    used = {int(bt[b, j]) for b, L_ in enumerate(lens) for j in range((L_ + 63) // 64)}
    for pid in range(kv.shape[0]):
        if pid not in used:
            kv[pid] = 0x7F
    case.kv_cache = kv
    out, lse = supported(L, impl, case.to("cuda"), 0)
    ro, rl = oracle_full(case)
    assert_parity(out, lse, ro, rl, what="garbage outside the visible history")


def test_out_of_range_page_id_and_seq_len_are_masked_and_reported(L, impl):
    """Device-resident indices are checked on the device: a page id out of range
    is not read (its positions drop out of the softmax) and a seq_len beyond the
    block table is treated as 0; each sets its device error code."""
    lens = [300, 200, 90]
    case = synth.make_decode_case(88, lens, 12, 1, extra_pages=2)
    bt = case.block_table.clone()
    bt[1, 1] = case.kv_cache.shape[0] + 7           # request 1, positions 64..127
    case.block_table = bt
    B = len(lens)
    out = torch.full((B, 1, 12, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((B, 1, 12), float("nan"), device="cuda")
    g = case.to("cuda")
    L.mla_decode_paged(g.q, g.kv_cache, g.kv_scale, g.block_table, g.seq_lens, 0, g.sm_scale, out, lse)
    torch.cuda.synchronize()
    assert L.mla_device_error() == 2
    for b in range(B):
        mask = np.ones(max(lens), dtype=np.uint8)
        if b == 1:
            mask[64:128] = 0
        bt_b = case.block_table[b:b + 1].clone()
        bt_b[bt_b >= case.kv_cache.shape[0]] = 0    # the oracle reads only kept positions
        ro, rl = oracle.decode(case.q[b:b + 1], case.kv_cache, case.kv_scale, bt_b,
                               case.seq_lens[b:b + 1], case.sm_scale, pos_mask=mask)
        assert_parity(out[b:b + 1], lse[b:b + 1], ro, rl, what=f"request {b} with a bad page id")
    # a seq_len beyond 64 * max_pages: that request reads nothing
    sl = case.seq_lens.clone()
    sl[2] = 64 * case.block_table.shape[1] + 1
    L.mla_decode_paged(g.q, g.kv_cache, g.kv_scale, case.block_table.cuda(), sl.cuda(), 0, g.sm_scale,
                       out, lse)
    torch.cuda.synchronize()
    err = L.mla_device_error()
    assert err in (2, 3)                               # the bad page of request 1 may report first
    assert torch.all(out[2] == 0) and torch.all(torch.isneginf(lse[2]))


def test_many_short_requests(L, impl):
    """A thousand requests of 32..200 positions in one call (1,000 grid rows of CTAs,
    12,000 merge rows when split).  (With a single visible position the answer is
    that position's value, up to ~4.5 in magnitude, where bf16 rounding alone
    exceeds the 1e-2 absolute bound; those cases are covered at small B.)"""
    rng = np.random.default_rng(1000)
    lens = [int(x) for x in rng.integers(32, 201, size=1000)]
    case = synth.make_decode_case(1000, lens, 12, 1)
    for n_splits in (0, 3):
        out, lse = supported(L, impl, case.to("cuda"), n_splits)
        ro, rl = oracle_full(case)
        assert_parity(out, lse, ro, rl, what=f"1,000 requests, splits={n_splits}")


def test_zero_query_heads_give_the_uniform_average(L, impl):
    """Heads whose query is all zero score every position 0: the answer is the plain
    mean of the visible values and lse = ln n (the oracle's closed-form pin)."""
    lens = [777, 64, 3]
    case = synth.make_decode_case(1001, lens, 16, 1)
    q = case.q.clone()
    q[:, :, 3] = 0
    q[:, :, 11] = 0
    case.q = q
    out, lse = supported(L, impl, case.to("cuda"), 0)
    ro, rl = oracle_full(case)
    assert_parity(out, lse, ro, rl, what="zero query heads")
    got = lse.cpu().numpy()[:, 0, [3, 11]]
    np.testing.assert_allclose(got, np.log(np.array(lens, dtype=np.float64))[:, None].repeat(2, 1),
                               atol=1e-4)


def test_lse_optional_and_deterministic(L, impl):
    case = synth.workload_case("tp8_batch", reduced=True).to("cuda")
    o1, l1 = supported(L, impl, case, 0)
    o2, _ = run(L, case, 0, with_lse=False)
    o3, l3 = run(L, case, 0)
    assert torch.equal(o1, o2) and torch.equal(o1, o3) and torch.equal(l1, l3)


def test_runs_on_a_side_stream(L, impl):
    case = synth.workload_case("tiny").to("cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        out, lse = supported(L, impl, case, 4)
    ro, rl = oracle_full(case)
    assert_parity(out, lse, ro, rl, what="side stream")


def test_graph_capture_and_replay_with_new_inputs(L, impl):
    """A serving loop captures the decode step once and replays it with new
    inputs written in place: each replay must answer for the inputs it sees."""
    lens = [700, 1500, 64]
    make = lambda seed: synth.make_decode_case(seed, lens, 12, 1, extra_pages=2)  # noqa: E731
    live = make(71).to("cuda")  # the buffers the graph is captured on
    out = torch.empty((3, 1, 12, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((3, 1, 12), device="cuda")
    s = torch.cuda.Stream()

    def call():
        L.mla_decode_paged(live.q, live.kv_cache, live.kv_scale, live.block_table, live.seq_lens, 0,
                           live.sm_scale, out, lse, s)

    with torch.cuda.stream(s):
        call()  # warm-up: the library's scratch for this stream exists before capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        call()
    for seed in (72, 71, 73):
        src = make(seed)
        for dst_t, src_t in ((live.q, src.q), (live.kv_cache, src.kv_cache), (live.kv_scale, src.kv_scale),
                             (live.block_table, src.block_table), (live.seq_lens, src.seq_lens)):
            dst_t.copy_(src_t)
        out.fill_(float("nan"))
        torch.cuda.synchronize()
        with torch.cuda.stream(s):
            g.replay()
        torch.cuda.synchronize()
        assert L.mla_device_error() == 0
        ro, rl = oracle_full(src)
        assert_parity(out, lse, ro, rl, what=f"graph replay, inputs of seed {seed}")


def _one_page_partitions(L, case, s, out, lse):
    """A call with one partition per page: a large split scratch (B x T x H
    rows x 2,052 bytes per partition)."""
    pages = case.block_table.shape[1]
    L.mla_decode_paged(case.q, case.kv_cache, case.kv_scale, case.block_table, case.seq_lens, pages,
                       case.sm_scale, out, lse, s)


@pytest.mark.filterwarnings("ignore:The CUDA Graph is empty")  # the refused capture records nothing
def test_capture_that_would_grow_the_scratch_is_refused(L):
    """A captured call may not allocate: if the stream's scratch is too small the
    call is refused with MLA_ERR_UNSUPPORTED and records nothing; after an
    uncaptured call of that size the same capture works and replays correctly.
    128 partitions x 4 x 128 rows need ~135 MB, more than any earlier call of
    the suite made any stream hold."""
    case = synth.make_decode_case(95, [8192, 8000, 5000, 8192], 128, 1).to("cuda")
    out = torch.full((4, 1, 128, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((4, 1, 128), float("nan"), device="cuda")
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    refused = False
    try:
        with torch.cuda.graph(g, stream=s):
            _one_page_partitions(L, case, s, out, lse)
    except L.MlaError as e:
        assert e.status == 2 and "capture" in str(e), e
        refused = True
    if refused:
        with torch.cuda.stream(s):
            _one_page_partitions(L, case, s, out, lse)  # uncaptured: the scratch grows
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            _one_page_partitions(L, case, s, out, lse)
    # else: this stream handle (streams are pooled) already held that much
    # scratch, so the first capture was valid; its replay is checked below
    out.fill_(float("nan"))
    lse.fill_(float("nan"))
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        g.replay()
    torch.cuda.synchronize()
    assert L.mla_device_error() == 0
    reqs, heads = [0, 2], [0, 77, 127]
    ro, rl = oracle_rows(case, reqs, heads)
    assert_parity(out[reqs][:, :, heads], lse[reqs][:, :, heads], ro, rl,
                  what="captured after the scratch grew, sampled rows")
    assert not torch.isnan(out).any() and not torch.isnan(lse).any()
    if not refused:
        pytest.skip("the stream already held enough scratch: the refusal was not exercised")


def test_graph_survives_a_later_larger_call(L):
    """The scratch a captured call used is retired, not freed, when a later
    uncaptured call on the stream needs more: replaying the graph afterwards
    still answers correctly."""
    lens = [1200, 3000]
    live = synth.make_decode_case(96, lens, 12, 1, extra_pages=2).to("cuda")
    out = torch.empty((2, 1, 12, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((2, 1, 12), device="cuda")
    s = torch.cuda.Stream()

    def call():
        L.mla_decode_paged(live.q, live.kv_cache, live.kv_scale, live.block_table, live.seq_lens, 0,
                           live.sm_scale, out, lse, s)

    with torch.cuda.stream(s):
        call()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        call()
    # 256 partitions x 4 x 128 rows (~270 MB): the stream's scratch must grow
    big = synth.make_decode_case(98, [16384] * 4, 128, 1).to("cuda")
    with torch.cuda.stream(s):
        _one_page_partitions(L, big, s, torch.empty((4, 1, 128, 512), dtype=torch.bfloat16, device="cuda"),
                             None)
    torch.cuda.synchronize()
    assert L.mla_device_error() == 0
    src = synth.make_decode_case(97, lens, 12, 1, extra_pages=2)
    for dst_t, src_t in ((live.q, src.q), (live.kv_cache, src.kv_cache), (live.kv_scale, src.kv_scale),
                         (live.block_table, src.block_table), (live.seq_lens, src.seq_lens)):
        dst_t.copy_(src_t)
    out.fill_(float("nan"))
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        g.replay()
    torch.cuda.synchronize()
    assert L.mla_device_error() == 0
    ro, rl = oracle_full(src)
    assert_parity(out, lse, ro, rl, what="graph replayed after the stream's scratch grew")


def test_release_graph_scratch_frees_what_captures_kept(L):
    """mla_release_graph_scratch frees the split scratch that captured calls used:
    the buffer a later growth retired and the one still attached to the stream.
    Once the graphs are destroyed, the device's free memory grows by about those
    bytes, the stream keeps working (its next call allocates anew) and a second
    release has nothing to do."""
    s = torch.cuda.Stream()
    small = synth.make_decode_case(99, [4096] * 4, 128, 1).to("cuda")   # 64 one-page partitions
    big = synth.make_decode_case(98, [16384] * 4, 128, 1).to("cuda")    # 256
    out = torch.empty((4, 1, 128, 512), dtype=torch.bfloat16, device="cuda")
    with torch.cuda.stream(s):
        _one_page_partitions(L, small, s, out, None)
    torch.cuda.synchronize()
    g1 = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g1, stream=s):
        _one_page_partitions(L, small, s, out, None)
    with torch.cuda.stream(s):  # grows the scratch: the captured buffer is retired
        _one_page_partitions(L, big, s, out, None)
    torch.cuda.synchronize()
    g2 = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g2, stream=s):  # the new buffer is now a graph's too
        _one_page_partitions(L, big, s, out, None)
    torch.cuda.synchronize()
    assert L.mla_device_error() == 0
    del g1, g2
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    L.mla_release_graph_scratch()
    torch.cuda.synchronize()
    free1 = torch.cuda.mem_get_info()[0]
    kept = 1.25 * (L.mla_decode_workspace_bytes(4, 1, 128, 64) + L.mla_decode_workspace_bytes(4, 1, 128, 256))
    assert free1 - free0 >= 0.5 * kept, (free0, free1, kept)
    lse = torch.empty((4, 1, 128), device="cuda")
    out.fill_(float("nan"))
    with torch.cuda.stream(s):
        L.mla_decode_paged(small.q, small.kv_cache, small.kv_scale, small.block_table, small.seq_lens, 5,
                           small.sm_scale, out, lse, s)
    torch.cuda.synchronize()
    assert L.mla_device_error() == 0
    ro, rl = oracle_full(small)
    assert_parity(out, lse, ro, rl, what="decode on a stream whose graph scratch was released")
    L.mla_release_graph_scratch()


def test_two_streams_at_once(L, impl):
    """Calls on two streams run concurrently with their own split scratch."""
    cases = [synth.make_decode_case(81 + k, [3000, 900], 12, 1).to("cuda") for k in range(2)]
    streams = [torch.cuda.Stream() for _ in range(2)]
    outs = [torch.full((2, 1, 12, 512), float("nan"), dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    lses = [torch.full((2, 1, 12), float("nan"), device="cuda") for _ in range(2)]
    torch.cuda.synchronize()
    for _ in range(3):
        for c, st, o, l in zip(cases, streams, outs, lses):
            with torch.cuda.stream(st):
                L.mla_decode_paged(c.q, c.kv_cache, c.kv_scale, c.block_table, c.seq_lens, 0, c.sm_scale,
                                   o, l, st)
    torch.cuda.synchronize()
    assert L.mla_device_error() == 0
    for k in range(2):
        ro, rl = oracle_full(synth.make_decode_case(81 + k, [3000, 900], 12, 1))
        assert_parity(outs[k], lses[k], ro, rl, what=f"stream {k}")


def test_dcp_shards_merge_to_unsharded(L, impl):
    """Section 1 (DCP): 8 contiguous shards of one history, each decoded on its own
    (out + lse), merged by mla_merge_partials, equal the unsharded oracle."""
    sc = synth.make_sharded_case(3, 2, 96, 1200, 8)
    outs, lses = [], []
    for sh in sc.shards:
        o, l = supported(L, impl, sh.to("cuda"), 0)
        ro, rl = oracle_full(sh)
        assert_parity(o, l, ro, rl, what="one shard")
        outs.append(o)
        lses.append(l)
    po, pl = torch.stack(outs), torch.stack(lses)
    out = torch.full(po.shape[1:], float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full(pl.shape[1:], float("nan"), dtype=torch.float32, device="cuda")
    L.mla_merge_partials(po, pl, 8, out, lse)
    torch.cuda.synchronize()
    ro, rl = oracle_full(sc.full)
    assert_parity(out, lse, ro, rl, what="merged shards vs unsharded")


def test_dcp_verify_shards_merge_to_unsharded(L, impl):
    """Multi-token verify through the DCP path (section 1): 4 contiguous shards of
    one history with T = 4 draft positions at its end.  Shards before the last
    are decoded as T = 1 calls with T*H rows (every draft query sees all of their
    positions); the last shard keeps T = 4 and the causal rule.  mla_merge_partials
    of the four (out, lse) equals the unsharded causal oracle."""
    T, H, n = 4, 12, 4
    sc = synth.make_sharded_case(19, 3, H, 4 * 700, n, T=T)
    outs, lses = [], []
    for s, sh in enumerate(sc.shards):
        g = sh.to("cuda")
        B = g.q.shape[0]
        if s < n - 1:
            g.q = g.q.reshape(B, 1, T * H, 576)
            o, l = supported(L, impl, g, 0)
            o, l = o.reshape(B, T, H, 512), l.reshape(B, T, H)
        else:
            o, l = supported(L, impl, g, 0)
        outs.append(o)
        lses.append(l)
    po, pl = torch.stack(outs), torch.stack(lses)
    out = torch.full(po.shape[1:], float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full(pl.shape[1:], float("nan"), dtype=torch.float32, device="cuda")
    L.mla_merge_partials(po, pl, n, out, lse)
    torch.cuda.synchronize()
    ro, rl = oracle_full(sc.full)
    assert_parity(out, lse, ro, rl, what="DCP verify: merged shards vs unsharded causal")


# ----------------------------------------------------------------------------
# mla_merge_partials on its own
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("S", [1, 2, 8, 32, 33, 100, 300, 1000])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_merge_partials_matches_oracle(L, S, dtype):
    g = torch.Generator().manual_seed(S)
    rows = (3, 5)
    # attention outputs are weighted averages of latents: |o| well below 1 (at |o| >= 4
    # bf16 rounding alone would exceed the 1e-2 absolute bound)
    po = (0.25 * torch.randn((S, *rows, 512), generator=g)).to(dtype)
    pl = (torch.randn((S, *rows), generator=g) * 3).float()
    drop = torch.rand((S, *rows), generator=g) < 0.3
    pl[drop] = float("-inf")
    pl[:, 0, 0] = float("-inf")  # a row with every shard empty
    empty = torch.isinf(pl)
    po_ref = po.clone()
    po_ref[empty] = 0
    po[empty] = float("nan")  # the values of an empty shard are ignored, whatever they hold
    out = torch.full((*rows, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full(rows, float("nan"), dtype=torch.float32, device="cuda")
    L.mla_merge_partials(po.cuda(), pl.cuda(), S, out, lse)
    torch.cuda.synchronize()
    ro, rl = oracle.merge(po_ref.float().numpy().astype(np.float64), pl.numpy().astype(np.float64))
    assert_parity(out, lse, ro, rl, what=f"merge S={S}")


@pytest.mark.parametrize("rows", [(40, 32), (12, 32)])
@pytest.mark.parametrize("S", [1, 3, 8, 19, 32])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_merge_partials_many_rows_matches_oracle(L, S, dtype, rows):
    """1,280 rows: the one-warp-per-row streaming path (DCP merges, large split
    combines); 384 rows: that path for bf16 parts, the (row, 64 dims) warps for
    fp32.  With empty parts and an all-empty row."""
    g = torch.Generator().manual_seed(100 + S)
    po = (0.25 * torch.randn((S, *rows, 512), generator=g)).to(dtype)
    pl = (torch.randn((S, *rows), generator=g) * 3).float()
    drop = torch.rand((S, *rows), generator=g) < 0.3
    pl[drop] = float("-inf")
    pl[:, 7, 9] = float("-inf")
    empty = torch.isinf(pl)
    po_ref = po.clone()
    po_ref[empty] = 0
    po[empty] = float("nan")
    out = torch.full((*rows, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full(rows, float("nan"), dtype=torch.float32, device="cuda")
    L.mla_merge_partials(po.cuda(), pl.cuda(), S, out, lse)
    torch.cuda.synchronize()
    ro, rl = oracle.merge(po_ref.float().numpy().astype(np.float64), pl.numpy().astype(np.float64))
    assert_parity(out, lse, ro, rl, what=f"merge S={S}, rows {rows}")


# ----------------------------------------------------------------------------
# Full-size workloads, launched as the benchmark launches them; sampled rows
# ----------------------------------------------------------------------------

FULL = {
    "tiny": ([0], list(range(12))),
    "tp8_batch": ([0, 5, 7], [0, 6, 11]),
    "verify": (None, [0, 11]),
    "long": ([0], [0, 7]),
    "ragged": (None, [3, 10]),
}


@pytest.mark.parametrize("name", sorted(FULL))
def test_full_size_sampled_rows(L, impl, name):
    """Each full-size workload at the count the benchmark plans from the host
    lengths (mla_plan_splits) and at the automatic count, where they differ."""
    case = synth.workload_case(name, device="cuda")
    if name == "tiny":
        counts = [4]
    else:
        mp = case.block_table.shape[1]
        counts = sorted({L.mla_plan_splits(case.B, case.T, case.H, case.lens, mp, 0),
                         L.mla_auto_splits(case.B, case.T, case.H, mp, 0)})
    reqs, heads = FULL[name]
    if reqs is None:  # shortest, longest and one in between
        order = np.argsort(case.lens)
        reqs = sorted({int(order[0]), int(order[len(order) // 2]), int(order[-1])})
    ro, rl = oracle_rows(case, reqs, heads)
    for n_splits in counts:
        out, lse = supported(L, impl, case, n_splits)
        o = out[reqs][:, :, heads]
        l = lse[reqs][:, :, heads]
        assert_parity(o, l, ro, rl, what=f"full {name}/{impl} splits={n_splits}")
        assert not torch.isnan(out).any() and not torch.isnan(lse).any()


def test_full_size_dcp_shards_and_merge(L, impl):
    sc = synth.make_sharded_case(3, 32, 96, 142000, 8, device="cuda")
    outs, lses = [], []
    for sh in sc.shards:
        o, l = supported(L, impl, sh, 0)
        outs.append(o)
        lses.append(l)
    reqs, heads = [0, 31], [0, 50, 95]
    ro, rl = oracle_rows(sc.shards[3], reqs, heads)
    assert_parity(outs[3][reqs][:, :, heads], lses[3][reqs][:, :, heads], ro, rl, what="shard 3")
    po, pl = torch.stack(outs), torch.stack(lses)
    out = torch.full(po.shape[1:], float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full(pl.shape[1:], float("nan"), dtype=torch.float32, device="cuda")
    L.mla_merge_partials(po, pl, 8, out, lse)
    torch.cuda.synchronize()
    ro, rl = oracle_rows(sc.full, reqs, heads)
    assert_parity(out[reqs][:, :, heads], lse[reqs][:, :, heads], ro, rl, what="merged 142,000")
    assert not torch.isnan(out).any()


# ----------------------------------------------------------------------------
# Longest-first launches (more CTAs than SMs, <= 1,024 requests): a one-CTA
# kernel orders all (request, partition) units longest first from the
# device-resident lengths; CTA k of the 12-head kernel takes entry k of that
# order, and the G row-CTAs k = G e .. G e + G - 1 of the wide kernel take
# entry e; the split combine counts the partitions past a history as empty
# ----------------------------------------------------------------------------

def _ragged(seed, B, lo, hi, zeros=0):
    rng = np.random.default_rng([seed, 23])
    lens = [int(x) for x in rng.integers(lo, hi, size=B)]
    for k in range(zeros):
        lens[(7 * k + 3) % B] = 0
    return lens


@pytest.mark.parametrize("B,H,T,n_splits,zeros,hi", [
    (20, 12, 1, 12, 0, 2600),    # 240 units of up to ~8 pages
    (64, 12, 1, 0, 5, 2600),     # automatic count, empty requests
    (40, 4, 4, 6, 2, 2600),      # 16 rows (causal verify), 240 units
    (256, 12, 1, 2, 9, 2600),
    (1024, 12, 1, 2, 30, 500),   # the largest longest-first batch
    (20, 12, 4, 6, 2, 2600),     # wide kernel: 48 rows (2 row-CTAs per unit), 240 CTAs
    (12, 96, 1, 5, 1, 4000),     # wide kernel: 96 rows (3 row-CTAs per unit), 180 CTAs
    (1025, 12, 1, 2, 0, 500),    # one more request: request order
    (160, 16, 1, 1, 0, 2600),    # unsplit: one CTA per request
])
def test_longest_first_launch_matches_oracle(L, impl, B, H, T, n_splits, zeros, hi):
    lens = _ragged(B + H + T, B, T, hi, zeros)
    case = synth.make_decode_case(3000 + B, lens, H, T, extra_pages=2)
    out, lse = supported(L, impl, case.to("cuda"), n_splits)
    ro, rl = oracle_full(case)
    assert_parity(out, lse, ro, rl, what=f"B={B} H={H} T={T} splits={n_splits}")


def test_longest_first_launch_repeated_and_replayed(L, impl):
    """Direct calls in a row and CUDA-graph replays of a longest-first launch all
    answer correctly (each launch recomputes its order from the lengths)."""
    lens = _ragged(77, 48, 1, 5000, 3)
    live = synth.make_decode_case(4001, lens, 12, 1, extra_pages=2).to("cuda")
    s = torch.cuda.Stream()
    out = torch.empty((48, 1, 12, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((48, 1, 12), device="cuda")

    def call():
        L.mla_decode_paged(live.q, live.kv_cache, live.kv_scale, live.block_table, live.seq_lens, 10,
                           live.sm_scale, out, lse, s)

    ro, rl = oracle_full(synth.make_decode_case(4001, lens, 12, 1, extra_pages=2))
    for _ in range(3):
        out.fill_(float("nan"))
        with torch.cuda.stream(s):
            call()
        torch.cuda.synchronize()
        assert L.mla_device_error() == 0
        assert_parity(out, lse, ro, rl, what="longest-first launch, direct call")
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        call()
    for _ in range(3):
        out.fill_(float("nan"))
        with torch.cuda.stream(s):
            g.replay()
        torch.cuda.synchronize()
        assert L.mla_device_error() == 0
        assert_parity(out, lse, ro, rl, what="longest-first launch, graph replay")


@pytest.mark.parametrize("lens", [
    [1000, 20000, 5, 0, 70000, 3000, 64, 9000],  # one wave of many short partitions
    "ragged32",                                   # a longest-first launch
])
def test_planned_split_counts_match_oracle(L, impl, lens):
    """The counts mla_plan_splits picks for uneven 12-head batches (85 partitions
    of 13 pages in one wave for the first; a multi-wave longest-first launch for
    the second) answer like the oracle."""
    if lens == "ragged32":
        lens = synth.ragged_lens(9, 32, 1024, 40000)
    case = synth.make_decode_case(4300 + len(lens), lens, 12, 1, extra_pages=1)
    n = L.mla_plan_splits(len(lens), 1, 12, lens, case.block_table.shape[1], 0)
    assert n > L.mla_auto_splits(len(lens), 1, 12, case.block_table.shape[1], 0)
    out, lse = supported(L, impl, case.to("cuda"), n)
    ro, rl = oracle_full(case)
    assert_parity(out, lse, ro, rl, what=f"planned {n} partitions")


def test_split_combine_ignores_partitions_past_each_history(L, impl):
    """The split combine counts a request's partitions past its history as empty
    whatever the scratch holds (a longest-first launch never writes them): a
    call whose requests are all long fills every partition of the stream's
    scratch with real partials, and the next call of the same shape on that
    stream, with mostly short requests, still answers exactly."""
    B, H, n_splits, hi = 48, 12, 10, 5120
    s = torch.cuda.Stream()
    full = synth.make_decode_case(4200, [hi] * B, H, 1).to("cuda")
    lens = [hi] + [int(x) for x in np.random.default_rng(4201).integers(1, 700, B - 1)]
    short = synth.make_decode_case(4202, lens, H, 1)
    g = short.to("cuda")
    assert g.block_table.shape == full.block_table.shape
    out = torch.empty((B, 1, H, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((B, 1, H), device="cuda")
    with torch.cuda.stream(s):
        L.mla_decode_paged(full.q, full.kv_cache, full.kv_scale, full.block_table, full.seq_lens, n_splits,
                           full.sm_scale, out, lse, s)
        out.fill_(float("nan"))
        L.mla_decode_paged(g.q, g.kv_cache, g.kv_scale, g.block_table, g.seq_lens, n_splits, g.sm_scale, out,
                           lse, s)
    torch.cuda.synchronize()
    assert L.mla_device_error() == 0
    ro, rl = oracle_full(short)
    assert_parity(out, lse, ro, rl, what="short requests after long ones on the same scratch")


def test_longest_first_launch_reports_a_bad_length(L):
    """A seq_len beyond the block table in a longest-first launch: that request
    reads nothing (out = 0, lse = -inf) and device error 3 is reported; the
    other requests are unaffected."""
    prev = L.mla_set_impl(IMPLS["tcgen05"])
    try:
        lens = _ragged(5, 30, 64, 3000)
        case = synth.make_decode_case(4100, lens, 12, 1)
        g = case.to("cuda")
        sl = g.seq_lens.clone()
        sl[4] = 64 * g.block_table.shape[1] + 5
        out = torch.full((30, 1, 12, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
        lse = torch.full((30, 1, 12), float("nan"), device="cuda")
        L.mla_decode_paged(g.q, g.kv_cache, g.kv_scale, g.block_table, sl, 8, g.sm_scale, out, lse)
        torch.cuda.synchronize()
        assert L.mla_device_error() == 3
        assert torch.all(out[4] == 0) and torch.all(torch.isneginf(lse[4]))
        keep = [b for b in range(30) if b != 4]
        ro, rl = oracle_full(case)
        assert_parity(out[keep], lse[keep], ro[keep], rl[keep], what="other requests")
    finally:
        L.mla_set_impl(prev)
