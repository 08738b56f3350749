"""The no-allocation entry point (mla_decode_paged_noalloc), through the C ABI.

Callers that must not have the library allocate device memory (an engine
that reserves the GPU's memory for its own page pool, or a latency-critical
step that must not pay for a first-use allocation) call this variant; its
split scratch is a fixed 8 MiB device array inside the library.  Its output
must agree with mla_decode_paged on the same inputs, on two calls in a row
(the array keeps the previous call's contents).  This file is collected last
so that a run stopping at the first failure has run every other test."""
import ctypes

import pytest
import torch

from mla_latent_kv_fp8_gb300 import synth
from tests.parity import assert_parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def L():
    from mla_latent_kv_fp8_gb300 import build
    build.build()
    from mla_latent_kv_fp8_gb300 import _lib
    _lib.lib()
    return _lib


def _outputs(case):
    B, T, H = case.q.shape[:3]
    out = torch.full((B, T, H, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((B, T, H), float("nan"), dtype=torch.float32, device="cuda")
    return out, lse


def _noalloc(L, case, n_splits, out, lse):
    """Direct C-ABI call of mla_decode_paged_noalloc (argument marshalling only)."""
    d = L.describe
    lib = L.lib()
    st = lib.mla_decode_paged_noalloc(
        ctypes.byref(d(case.q)), ctypes.byref(d(case.kv_cache)),
        ctypes.c_void_p(case.kv_scale.data_ptr()), ctypes.byref(d(case.block_table)),
        ctypes.byref(d(case.seq_lens)), int(n_splits), float(case.sm_scale),
        ctypes.byref(d(out)), ctypes.byref(d(lse)),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return st


@pytest.mark.parametrize("name,n_splits", [("tp8_batch", 0), ("verify", 5), ("tiny", 4)])
def test_noalloc_matches_allocating_entry_point_twice(L, name, n_splits):
    case = synth.workload_case(name, reduced=True).to("cuda")
    ref_out, ref_lse = _outputs(case)
    L.mla_decode_paged(case.q, case.kv_cache, case.kv_scale, case.block_table, case.seq_lens,
                       n_splits, case.sm_scale, ref_out, ref_lse)
    torch.cuda.synchronize()
    for _ in range(2):  # the fixed array keeps the previous call's contents
        out, lse = _outputs(case)
        assert _noalloc(L, case, n_splits, out, lse) == 0, L.mla_last_error()
        torch.cuda.synchronize()
        assert L.mla_device_error() == 0
        assert_parity(out, lse, ref_out.double().cpu().numpy(), ref_lse.double().cpu().numpy(),
                      what=f"no-allocation entry point, {name}")
    # the split scratch really was used
    assert L.mla_decode_workspace_bytes(case.B, case.T, case.H, 2) > 0


def test_noalloc_rejects_scratch_beyond_its_array(L):
    case = synth.make_decode_case(9, [64 * 4096], 12, 1, device="cuda")
    out, lse = _outputs(case)
    # 4096 partitions x 12 rows x 513 floats exceed the 8 MiB array
    st = _noalloc(L, case, 4096, out, lse)
    assert st == 2
    assert "exceeds" in L.mla_last_error()
