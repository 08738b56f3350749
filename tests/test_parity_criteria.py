"""The parity criteria themselves (CPU): the bf16 rounding allowance and the
magnitude-aware LSE bound."""
import numpy as np
import torch

from tests import parity


def test_bf16_half_ulp_matches_torch_rounding():
    rng = np.random.default_rng(3)
    x = np.concatenate([rng.standard_normal(20000) * s for s in (1e-3, 1.0, 10.0, 300.0)])
    r = torch.from_numpy(x).to(torch.bfloat16).double().numpy()
    # rounding to bf16 never moves a value by more than half an ulp ...
    assert np.all(np.abs(r - x) <= parity.bf16_half_ulp(x) * (1 + 1e-12))
    # ... and the allowance is tight: some values move by almost that much
    assert np.max(np.abs(r - x) / parity.bf16_half_ulp(x)) > 0.99


def test_exact_answer_rounded_to_bf16_passes_and_a_real_error_fails():
    rng = np.random.default_rng(4)
    ref = rng.standard_normal((2, 1, 3, 512)) * 2.5  # |ref| up to ~10: bf16 rounding > 1e-2 there
    lse = rng.standard_normal((2, 1, 3)) * 3
    out = torch.from_numpy(ref).to(torch.bfloat16)
    assert np.abs(out.double().numpy() - ref).max() > 1e-2  # the literal bound alone would fail
    parity.assert_parity(out, torch.from_numpy(lse).float(), ref, lse)
    ref2 = ref.copy()
    ref2[0, 0, 0, 5] = 0.5
    bad = ref2.copy()
    bad[0, 0, 0, 5] = 0.5 + 0.02  # 2e-2 off at |ref| = 0.5: beyond 1e-2 + 2^-10
    e = parity.errors(torch.from_numpy(bad).to(torch.bfloat16), torch.from_numpy(lse).float(), ref2, lse)
    assert e["out_bound_used"] > 1.0


def test_lse_bound_is_absolute_then_relative():
    assert parity.lse_bound(np.array([5.0]))[0] == 1e-4
    assert parity.lse_bound(np.array([-50.0]))[0] == 1e-4
    assert abs(parity.lse_bound(np.array([400.0]))[0] - 400 * 2.0 ** -20) < 1e-12
    # fp32 can hold the bound: its spacing at |lse| stays well below the bound
    for v in (1.0, 100.0, 1000.0, 1e5):
        assert np.spacing(np.float32(v)) * 4 <= parity.lse_bound(np.array([v]))[0]
