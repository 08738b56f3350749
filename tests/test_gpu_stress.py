"""GPU parity on inputs that drive the tensor-core kernels' own approximations
into their hard regimes, element by element against the FP64 oracle.

The tcgen05 kernels take each row's probabilities against a lazy reference
maximum (moved, with an in-place rescale of the accumulated output in tensor
memory, only when a score would exceed it by 8.8 log2 units), store them as two
e4m3 terms, and split the query into two exact e4m3 terms.  N(0,1) inputs give
flat softmaxes that rarely move the reference, so these cases plant structure
(mla_latent_kv_fp8_gb300.synth stress patterns):

  * peaked softmax: queries x4, x16, x64;
  * scores climbing across every partition, so the reference moves again and
    again after a warpgroup's first page (a device counter proves the rescale
    path ran), with the largest score on a partition's last page;
  * one dominant first position with every later score >= 20 log2 units below
    (the flushing of tiny probabilities), and its coherent worst case: ten
    thousand identical positions 15-20 log2 units below the peak, whose
    rounding errors all point the same way;
  * query rows with one outlier channel 1,024 times the others (scores of the
    usual size, so the elements 2^-10 below the row's maximum matter);
  * a tiny kv_scale (2^-20, with 10^4-times queries) and a large one (16, codes
    in e4m3's subnormal range).

Each runs on the 12-head kernel (H*T <= 16) and on the wide kernel (96 heads,
or 12 heads x 4 causal draft positions), with one partition, explicit counts
and the automatic count; reduced sizes compare every row, the full-size
workloads sampled rows.  The CUDA-core kernel runs the same cases."""
import numpy as np
import pytest
import torch

import oracle
from mla_latent_kv_fp8_gb300 import synth
from tests.parity import assert_parity
from tests.test_gpu_parity import IMPLS, oracle_full, oracle_rows, supported  # noqa: F401

pytestmark = pytest.mark.gpu


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


def counted(L, case, n_splits):
    """One decode with the rescale counters armed: (out, lse, [rescales after a
    warpgroup's first page, reference moves])."""
    counts = torch.zeros(2, dtype=torch.int32, device="cuda")
    L.mla_test_count_rescales(counts)
    out, lse = supported(L, None, case, n_splits)
    return out, lse, counts.cpu().tolist()


def case_of(seed, lens, H, T, pattern, device="cpu"):
    return synth.make_decode_case(seed, lens, H, T, pattern=pattern, device=device, extra_pages=2)


SHAPES = {  # name: (H, T) -- 12-head kernel, wide kernel (96 heads), wide causal verify
    "12h": (12, 1),
    "96h": (96, 1),
    "verify": (12, 4),
}


# ----------------------------------------------------------------------------
# Reduced sizes: every row
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("shape", sorted(SHAPES))
@pytest.mark.parametrize("gain", [4, 16, 64])
def test_peaked_softmax(L, impl, shape, gain):
    H, T = SHAPES[shape]
    case = case_of(200 + gain, [3000, 777, 64], H, T, synth.PeakedQueries(gain))
    ro, rl = oracle_full(case)
    for n_splits in (1, 5, 0):
        out, lse = supported(L, impl, case.to("cuda"), n_splits)
        assert_parity(out, lse, ro, rl, what=f"q x{gain} {shape} splits={n_splits}")


@pytest.mark.parametrize("shape", sorted(SHAPES))
@pytest.mark.parametrize("n_splits", [1, 3])
def test_scores_climbing_across_partitions(L, impl, shape, n_splits):
    """Scores rise by ~60 log2 units over every partition (the planted amplitude
    restarts at each partition's first position), so each partition's maximum is
    on its last page and the running reference moves every few pages."""
    H, T = SHAPES[shape]
    lens = [6400, 5000, 4100]
    chunk_pos = 64 * L.mla_split_chunk_pages(100, n_splits)  # partitions of the 100-page table
    case = case_of(300 + n_splits, lens, H, T, synth.ClimbingKeys(72.0, chunk_pos))
    case.block_table = torch.nn.functional.pad(case.block_table, (0, 100 - case.block_table.shape[1]))
    ro, rl = oracle_full(case)
    g = case.to("cuda")
    if impl == "tcgen05":
        out, lse, (rescales, moves) = counted(L, g, n_splits)
        # every partition of every request climbs: many moves after the first page
        assert rescales >= 10 * n_splits * len(lens), (rescales, moves)
        assert moves > rescales
    else:
        out, lse = supported(L, impl, g, n_splits)
    assert_parity(out, lse, ro, rl, what=f"climbing {shape} splits={n_splits}")


@pytest.mark.parametrize("shape", sorted(SHAPES))
def test_one_dominant_position_and_a_flushed_tail(L, impl, shape):
    """Position 0 scores 28+ log2 units above every other position: the others'
    probabilities fall below e4m3's range and are flushed; the answer is position
    0's value and its lse."""
    H, T = SHAPES[shape]
    case = case_of(400, [10240, 3000, 65], H, T, synth.FirstPeak(40.0))
    ro, rl = oracle_full(case)
    for n_splits in (1, 4, 0):
        out, lse = supported(L, impl, case.to("cuda"), n_splits)
        assert_parity(out, lse, ro, rl, what=f"first peak {shape} splits={n_splits}")


@pytest.mark.parametrize("shape", ["12h", "96h"])
@pytest.mark.parametrize("n_splits", [1, 2])
def test_coherent_tail_below_a_peak(L, impl, shape, n_splits):
    """10,240 identical positions 15-20 log2 units below one peak, in one
    partition (n_splits = 1) or two: every tail probability carries the same
    rounding error, so a relative error of the probability encoding at that
    depth shows up undiluted in the answer."""
    H, T = SHAPES[shape]
    amps = [19.0, 20.5, 21.6, 22.5, 24.0]
    case = case_of(500, [10241] * len(amps), H, T, synth.CoherentTail(amps))
    ro, rl = oracle_full(case)
    out, lse = supported(L, impl, case.to("cuda"), n_splits)
    assert_parity(out, lse, ro, rl, what=f"coherent tail {shape} splits={n_splits}")


@pytest.mark.parametrize("shape", sorted(SHAPES))
def test_outlier_query_channels(L, impl, shape):
    H, T = SHAPES[shape]
    case = case_of(600, [2500, 130], H, T, synth.OutlierQueries(1024.0, 16.0))
    ro, rl = oracle_full(case)
    for n_splits in (1, 0):
        out, lse = supported(L, impl, case.to("cuda"), n_splits)
        assert_parity(out, lse, ro, rl, what=f"outlier q {shape} splits={n_splits}")


@pytest.mark.parametrize("shape", sorted(SHAPES))
@pytest.mark.parametrize("which", ["tiny", "large"])
def test_extreme_kv_scale(L, impl, shape, which):
    """tiny: latents x 1e-4 quantised with kv_scale = 2^-20 and queries x 1e4
    (scores of the usual size, answers ~1e-4: the relative bound carries the
    check); large: kv_scale = 16 with codes in e4m3's subnormal range and
    queries / 16."""
    H, T = SHAPES[shape]
    pat = (synth.ScaledCache(1e-4, 2.0 ** -20, 1e4) if which == "tiny"
           else synth.ScaledCache(1.0, 16.0, 1.0 / 16.0))
    case = case_of(700, [2000, 333], H, T, pat)
    ro, rl = oracle_full(case)
    for n_splits in (1, 0):
        out, lse = supported(L, impl, case.to("cuda"), n_splits)
        e = assert_parity(out, lse, ro, rl, what=f"kv_scale {which} {shape} splits={n_splits}")
        assert e["rel_out"] <= 1.6e-2


# ----------------------------------------------------------------------------
# Full-size workloads with stressed inputs, launched as the benchmark launches
# them (automatic or planned split counts); sampled rows
# ----------------------------------------------------------------------------

def _full(name, pattern):
    seed = synth.WORKLOADS[name][1]
    if name == "tp8_batch":
        return synth.make_decode_case(seed, synth.tp8_lens(seed), 12, 1, device="cuda", pattern=pattern)
    if name == "long":
        return synth.make_decode_case(seed, [393216], 12, 1, device="cuda", pattern=pattern)
    if name == "dcp_shard":
        return synth.make_decode_case(seed, [17750] * 32, 96, 1, device="cuda", pattern=pattern)
    if name == "verify":
        return synth.make_decode_case(seed, synth.verify_lens(seed), 12, 4, device="cuda", pattern=pattern)
    raise KeyError(name)


FULL_ROWS = {"tp8_batch": ([0, 7], [0, 1, 6]), "long": ([0], [0, 1, 10]),
             "dcp_shard": ([0, 31], [0, 1, 95]), "verify": ([0, 15], [0, 1, 11])}


@pytest.mark.parametrize("name", sorted(FULL_ROWS))
@pytest.mark.parametrize("kind", ["climb", "peaked"])
def test_full_size_stressed(L, name, kind):
    """The full-size workloads with climbing scores (period = the automatic
    partition length, so every partition climbs to its last page) or queries
    x16, on the tensor-core kernels with the automatic split count."""
    prev = L.mla_set_impl(IMPLS["tcgen05"])
    try:
        seed = synth.WORKLOADS[name][1]
        if kind == "climb":
            lens = {"tp8_batch": synth.tp8_lens(seed), "long": [393216], "dcp_shard": [17750] * 32,
                    "verify": synth.verify_lens(seed)}[name]
            H, T = {"tp8_batch": (12, 1), "long": (12, 1), "dcp_shard": (96, 1), "verify": (12, 4)}[name]
            mp = max(-(-x // 64) for x in lens)
            chunk = L.mla_split_chunk_pages(mp, L.mla_auto_splits(len(lens), T, H, mp, 0))
            pattern = synth.ClimbingKeys(72.0, 64 * chunk)
        else:
            pattern = synth.PeakedQueries(16.0)
        case = _full(name, pattern)
        out, lse, (rescales, moves) = counted(L, case, 0)
        if kind == "climb":
            assert rescales > 0, (rescales, moves)
        reqs, heads = FULL_ROWS[name]
        ro, rl = oracle_rows(case, reqs, heads)
        assert_parity(out[reqs][:, :, heads], lse[reqs][:, :, heads], ro, rl, what=f"full {name} {kind}")
        assert not torch.isnan(out).any() and not torch.isnan(lse).any()
    finally:
        L.mla_set_impl(prev)


def test_rescale_counter_is_one_shot_and_quiet_on_flat_inputs(L):
    """The counter hook applies to the next call only; flat N(0,1) inputs move
    each reference at the first page and almost never again."""
    prev = L.mla_set_impl(IMPLS["tcgen05"])
    try:
        case = synth.workload_case("tp8_batch", reduced=True).to("cuda")
        counts = torch.zeros(2, dtype=torch.int32, device="cuda")
        L.mla_test_count_rescales(counts)
        supported(L, None, case, 1)
        first = counts.cpu().tolist()
        supported(L, None, case, 1)  # not counted
        assert counts.cpu().tolist() == first
        assert first[1] >= case.B * 2  # every warpgroup sets its reference once
    finally:
        L.mla_set_impl(prev)
