"""Host-side logic of bench.py that needs no GPU: the shard plan of the DCP
multi-token verify measurement."""
import numpy as np
import pytest
import torch

import bench
from mla_latent_kv_fp8_gb300 import synth


@pytest.mark.parametrize("n_sh", [2, 8])
def test_dcp_verify_plan_covers_each_history_once(n_sh):
    lens = synth.verify_lens(4)  # the verify workload's contexts
    B, T = len(lens), 4
    max_pages = -(-max(lens) // 64)
    bt = torch.stack([torch.randperm(10 * max_pages)[:max_pages] for _ in range(B)]).to(torch.int32)
    plan = bench.dcp_verify_plan(lens, bt, n_sh, T)
    assert len(plan) == n_sh
    for b, L in enumerate(lens):
        pages, pos = [], 0
        for s, (table, sl) in enumerate(plan):
            n = int(sl[b])
            if s < n_sh - 1:
                assert n % 64 == 0  # shards start on page boundaries
            np_ = -(-n // 64)
            pages += table[b, :np_].tolist()
            pos += n
        assert pos == L  # the shards tile the history exactly
        assert pages == bt[b, :-(-L // 64)].tolist()  # in order, each page once
        assert int(plan[-1][1][b]) >= T  # the draft positions lie in the last shard


def test_dcp_verify_plan_rejects_short_histories():
    bt = torch.arange(4, dtype=torch.int32).reshape(1, 4)
    with pytest.raises(ValueError):
        bench.dcp_verify_plan([7 * 64 + 2], bt, 8, 4)


def test_parity_of_applies_the_tolerances():
    ro = np.zeros((2, 1, 3, 512))
    ro[0] = 0.5
    rl = np.array([[[1.0, 2.0, 3.0]], [[-np.inf] * 3]])
    o, l = ro.copy(), rl.copy()
    assert bench.parity_of(o, l, ro, rl)["pass"]
    o2 = o.copy()
    o2[0, 0, 1, 7] += 0.011  # above the 1e-2 absolute bound
    assert not bench.parity_of(o2, l, ro, rl)["pass"]
    l2 = l.copy()
    l2[0, 0, 2] += 2e-4  # above the 1e-4 LSE bound
    assert not bench.parity_of(o, l2, ro, rl)["pass"]
    o3 = o.copy()
    o3[1, 0, 0, 0] = 1e-3  # an empty row must be exactly 0
    assert not bench.parity_of(o3, l, ro, rl)["pass"]
    o4 = o.copy()
    o4[0, 0, 0, 0] = np.nan
    assert not bench.parity_of(o4, l, ro, rl)["pass"]


def test_algorithmic_flops_counts_visible_positions():
    # T = 1: every row sees the whole history
    assert bench.algorithmic_flops([100, 0, 64], 1, 12) == 2176 * 12 * 164
    # causal verify: query t of a length-L request sees L - T + 1 + t positions
    lens, T, H = [50, 7], 4, 3
    brute = sum(2176 * H * (L - T + 1 + t) for L in lens for t in range(T))
    assert bench.algorithmic_flops(lens, T, H) == brute


def test_tensor_roofline_fields():
    r = bench.tensor_roofline(1e12, 1e-3)  # 1 TFLOP in 1 ms
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s"
    assert abs(r["achieved"] - 1000.0) < 1e-6
    assert abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-3
