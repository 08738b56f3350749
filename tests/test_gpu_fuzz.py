"""Seeded random shapes against the FP64 oracle, for both kernel families:
request count, heads, draft positions (causal), ragged lengths (empty ones
included) and split counts (automatic and explicit) drawn at random, so that
the row-group, partition and masking boundaries are hit in combinations the
hand-picked cases do not list."""
import numpy as np
import pytest

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


@pytest.mark.parametrize("seed", range(24))
def test_random_shapes_match_oracle(L, impl, seed):
    lens, H, T, n_splits = _draw(seed)
    case = synth.make_decode_case(5000 + seed, lens, H, T, extra_pages=int(seed % 3))
    out, lse = supported(L, impl, case.to("cuda"), n_splits)
    ro, rl = oracle.decode(case.q, case.kv_cache, case.kv_scale, case.block_table, case.seq_lens,
                           case.sm_scale)
    assert_parity(out, lse, ro, rl, what=f"seed {seed}: lens={lens} H={H} T={T} splits={n_splits}")
