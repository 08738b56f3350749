"""Host-side logic of bench.py that needs no GPU: parity bookkeeping, flop
counts, the tensor roofline and the gate on recorded ncu counters."""
import numpy as np
import pytest
import torch

import bench
from mla_latent_kv_fp8_gb300 import synth


def test_dcp_verify_plan_rejects_short_histories():
    from mla_latent_kv_fp8_gb300.dcp import shard_plan
    bt = torch.arange(4, dtype=torch.int32).reshape(1, 4)
    with pytest.raises(ValueError):
        shard_plan([7 * 64 + 2], bt, 8, 4)


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


def test_device_code_digest_ignores_comments_and_host_code(tmp_path, monkeypatch):
    """The ncu traffic record stays valid across comment and host-side edits of a
    kernel file and is invalidated by any change to its device code."""
    root = tmp_path
    (root / "k.cu").write_text("__global__ void k(int* p) {\n    p[0] = 1;  // store\n}\n"
                               + bench.HOST_SIDE_MARKER + "\nint launch() { return 0; }\n")
    monkeypatch.setattr(bench, "ROOT", str(root))
    d0 = bench.device_code_digest(["k.cu"])
    (root / "k.cu").write_text("// a new header comment\n\n__global__ void k(int* p) {\n    p[0] = 1;  // the store\n}\n"
                               + bench.HOST_SIDE_MARKER + "\nint launch() { return 1; }\n")
    assert bench.device_code_digest(["k.cu"]) == d0
    (root / "k.cu").write_text("__global__ void k(int* p) {\n    p[0] = 2;\n}\n" + bench.HOST_SIDE_MARKER + "\n")
    assert bench.device_code_digest(["k.cu"]) != d0


def test_ncu_traffic_record_is_gated_on_the_device_code():
    import json
    import os
    p = os.path.join(bench.ROOT, "profiles", "ncu_traffic.json")
    with open(p) as f:
        d = json.load(f)
    for key, e in d.items():
        if key.startswith("_"):
            continue
        fam, workload = key.split("/")
        r = bench.ncu_traffic(fam, workload)
        current = e.get("device_code_digest") == bench.device_code_digest(bench.KERNEL_SOURCES[fam])
        assert (r is not None) == current, key
        if r is not None:
            assert r["dram_bytes_per_launch"] == e["dram_bytes_per_launch"]
