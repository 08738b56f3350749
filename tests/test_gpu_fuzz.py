"""Seeded random shapes against the FP64 oracle, for both kernel families:
request count, heads, draft positions (causal), ragged lengths (empty ones
included) and split counts (automatic and explicit) drawn at random, so that
the kernel choice (16 rows per CTA, or 32-row CTAs sharing pages), partition
and masking boundaries are hit in combinations the hand-picked cases do not
list; and random merges (part counts, row counts, dtypes, empty parts) across
the three merge kernels."""
import numpy as np
import pytest
import torch

import oracle
from mla_latent_kv_fp8_gb300 import synth
from tests.parity import assert_parity
from tests.test_gpu_parity import IMPLS, supported  # noqa: F401  (fixtures below)

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


def _draw(seed):
    rng = np.random.default_rng([seed, 17])
    T = int(rng.choice([1, 1, 1, 2, 3, 4, 8]))
    H = int(rng.integers(1, 128 // T + 1))
    B = int(rng.integers(1, 5))
    lens = [int(x) for x in rng.integers(T, 2500, size=B)]
    if B > 1 and rng.random() < 0.3:
        lens[int(rng.integers(0, B))] = 0
    n_splits = int(rng.choice([0, 0, 1, int(rng.integers(2, 24))]))
    return lens, H, T, n_splits


@pytest.mark.parametrize("seed", range(48))
def test_random_shapes_match_oracle(L, impl, seed):
    lens, H, T, n_splits = _draw(seed)
    case = synth.make_decode_case(5000 + seed, lens, H, T, extra_pages=int(seed % 3))
    out, lse = supported(L, impl, case.to("cuda"), n_splits)
    ro, rl = oracle.decode(case.q, case.kv_cache, case.kv_scale, case.block_table, case.seq_lens,
                           case.sm_scale)
    assert_parity(out, lse, ro, rl, what=f"seed {seed}: lens={lens} H={H} T={T} splits={n_splits}")


def _draw_multiwave(seed):
    """Batches whose launches have more CTAs than SMs: the longest-first order
    of both kernels, at the planned, the automatic and random split counts."""
    rng = np.random.default_rng([seed, 29])
    T = int(rng.choice([1, 1, 2, 4]))
    H = int(rng.choice([int(rng.integers(1, 16 // T + 1)), int(rng.integers(16 // T + 1, 128 // T + 1))]))
    B = int(rng.integers(20, 49))
    lens = [int(x) for x in rng.integers(T, int(rng.choice([700, 1500])), size=B)]
    for k in range(int(rng.integers(0, 4))):
        lens[int(rng.integers(0, B))] = 0
    mode = seed % 3
    return lens, H, T, mode, int(rng.integers(4, 13))


@pytest.mark.parametrize("seed", range(18))
def test_random_multiwave_launches_match_oracle(L, impl, seed):
    lens, H, T, mode, explicit = _draw_multiwave(seed)
    case = synth.make_decode_case(6000 + seed, lens, H, T, extra_pages=int(seed % 2))
    mp = case.block_table.shape[1]
    n_splits = (L.mla_plan_splits(len(lens), T, H, lens, mp, 0), 0, explicit)[mode]
    out, lse = supported(L, impl, case.to("cuda"), n_splits)
    ro, rl = oracle.decode(case.q, case.kv_cache, case.kv_scale, case.block_table, case.seq_lens,
                           case.sm_scale)
    assert_parity(out, lse, ro, rl, what=f"seed {seed}: B={len(lens)} H={H} T={T} splits={n_splits}")


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("seed", range(16))
def test_random_merges_match_oracle(L, seed, dtype):
    rng = np.random.default_rng([seed, 29])
    S = int(rng.choice([1, 2, 5, 8, 19, 32, 33, 64, 150]))
    rows = int(rng.choice([1, 7, 96, 255, 256, 700, 1216, 1500, 2000, 3072]))
    if S > 32:
        rows = min(rows, 700)  # keeps the host-side arrays small
    g = torch.Generator().manual_seed(9000 + seed)
    po = (0.25 * torch.randn((S, rows, 512), generator=g)).to(dtype)
    pl = (torch.randn((S, rows), generator=g) * 4).float()
    pl[torch.rand((S, rows), generator=g) < float(rng.choice([0.0, 0.2, 0.9]))] = float("-inf")
    empty = torch.isinf(pl)
    po_ref = po.clone()
    po_ref[empty] = 0
    po[empty] = float("nan")  # never-written parts must not leak into the answer
    out = torch.full((rows, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((rows,), float("nan"), dtype=torch.float32, device="cuda")
    L.mla_merge_partials(po.cuda(), pl.cuda(), S, out, lse)
    torch.cuda.synchronize()
    ro, rl = oracle.merge(po_ref.float().numpy().astype(np.float64), pl.numpy().astype(np.float64))
    assert_parity(out, lse, ro, rl, what=f"seed {seed}: S={S} rows={rows} {dtype}")
