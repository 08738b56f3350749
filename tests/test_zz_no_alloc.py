"""The no-allocation entry point (mla_decode_paged_noalloc), through the C ABI.

Callers that must not have the library allocate device memory (an engine
that reserves the GPU's memory for its own page pool, or a latency-critical
step that must not pay for a first-use allocation) call this variant; its
split scratch is a fixed 8 MiB device array inside the library.  Its output
must agree with the FP64 oracle, and with mla_decode_paged, on the same inputs,
on two calls in a row (the array keeps the previous call's contents), with the
call really split into several partitions.  This file is collected last so
that a run stopping at the first failure has run every other test."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from mla_latent_kv_fp8_gb300 import synth
from tests.parity import assert_parity

pytestmark = pytest.mark.gpu

ARRAY_BYTES = 8 << 20


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


def _noalloc(L, case, n_splits, out, lse, stream=None):
    """Direct C-ABI call of mla_decode_paged_noalloc (argument marshalling only)."""
    d = L.describe
    lib = L.lib()
    s = stream if stream is not None else torch.cuda.current_stream()
    return lib.mla_decode_paged_noalloc(
        ctypes.byref(d(case.q)), ctypes.byref(d(case.kv_cache)),
        ctypes.c_void_p(case.kv_scale.data_ptr()), ctypes.byref(d(case.block_table)),
        ctypes.byref(d(case.seq_lens)), int(n_splits), float(case.sm_scale),
        ctypes.byref(d(out)), ctypes.byref(d(lse)), ctypes.c_void_p(s.cuda_stream))


def _resolved_splits(L, case, n_splits):
    mp = case.block_table.shape[1]
    req = n_splits if n_splits > 0 else L.mla_auto_splits(case.B, case.T, case.H, mp, 0)
    chunk = L.mla_split_chunk_pages(mp, req)
    return -(-mp // chunk)


def _longest_first_case():
    """40 requests x 12 heads in 8 partitions: 320 units, more than SMs, so the
    12-head kernel takes them in longest-first order."""
    rng = np.random.default_rng(41)
    return synth.make_decode_case(4200, [int(x) for x in rng.integers(200, 3000, size=40)], 12, 1)


@pytest.mark.parametrize("name,n_splits", [("tp8_batch", 0), ("verify", 5), ("tiny", 4), ("longest_first", 8)])
def test_noalloc_matches_oracle_and_allocating_entry_point_twice(L, name, n_splits):
    cpu = _longest_first_case() if name == "longest_first" else synth.workload_case(name, reduced=True)
    case = cpu.to("cuda")
    n_eff = _resolved_splits(L, case, n_splits)
    assert n_eff > 1, "the case must use the split scratch"
    assert L.mla_decode_workspace_bytes(case.B, case.T, case.H, n_eff) <= ARRAY_BYTES
    ro, rl = oracle.decode(cpu.q, cpu.kv_cache, cpu.kv_scale, cpu.block_table, cpu.seq_lens, cpu.sm_scale)
    ref_out, ref_lse = _outputs(case)
    L.mla_decode_paged(case.q, case.kv_cache, case.kv_scale, case.block_table, case.seq_lens,
                       n_splits, case.sm_scale, ref_out, ref_lse)
    torch.cuda.synchronize()
    for _ in range(2):  # the fixed array keeps the previous call's contents
        out, lse = _outputs(case)
        assert _noalloc(L, case, n_splits, out, lse) == 0, L.mla_last_error()
        torch.cuda.synchronize()
        assert L.mla_device_error() == 0
        assert_parity(out, lse, ro, rl, what=f"no-allocation entry point vs oracle, {name}")
        # the same kernels and the same partition count: the same answer
        assert torch.equal(out, ref_out) and torch.equal(lse, ref_lse)


def test_noalloc_allocates_nothing(L):
    """Captured in global mode, any cudaMalloc / cudaFree of the call, or growth of
    the library's pooled scratch (which the library refuses during capture), would
    fail the capture; the captured call must also answer correctly."""
    cpu = synth.workload_case("tp8_batch", reduced=True)
    case = cpu.to("cuda")
    assert _resolved_splits(L, case, 0) > 1
    out, lse = _outputs(case)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        assert _noalloc(L, case, 0, out, lse, s) == 0, L.mla_last_error()  # per-device set-up
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        st = _noalloc(L, case, 0, out, lse, s)
    assert st == 0, L.mla_last_error()
    out.fill_(float("nan"))
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        g.replay()
    torch.cuda.synchronize()
    assert L.mla_device_error() == 0
    ro, rl = oracle.decode(cpu.q, cpu.kv_cache, cpu.kv_scale, cpu.block_table, cpu.seq_lens, cpu.sm_scale)
    assert_parity(out, lse, ro, rl, what="no-allocation entry point, captured")


def test_noalloc_automatic_count_fits_the_array(L):
    """n_splits = 0 caps the automatic count at what 8 MiB holds: 32 requests x 96
    heads over 30 pages want 3 partitions of 3,072 rows (18 MB); the call runs
    unsplit (2 partitions would already need 12.6 MB)."""
    cpu = synth.make_decode_case(91, [1900] * 32, 96, 1)
    case = cpu.to("cuda")
    assert L.mla_decode_workspace_bytes(32, 1, 96, _resolved_splits(L, case, 0)) > ARRAY_BYTES
    out, lse = _outputs(case)
    assert _noalloc(L, case, 0, out, lse) == 0, L.mla_last_error()
    torch.cuda.synchronize()
    assert L.mla_device_error() == 0
    reqs = [0, 17, 31]
    ro, rl = oracle.decode(cpu.q[reqs], cpu.kv_cache, cpu.kv_scale, cpu.block_table[reqs], cpu.seq_lens[reqs],
                           cpu.sm_scale)
    assert_parity(out[reqs], lse[reqs], ro, rl, what="no-allocation entry point, capped automatic count")


def test_noalloc_rejects_explicit_scratch_beyond_its_array(L):
    case = synth.make_decode_case(9, [64 * 4096], 12, 1, device="cuda")
    out, lse = _outputs(case)
    # 4096 partitions x 12 rows x 513 floats exceed the 8 MiB array
    st = _noalloc(L, case, 4096, out, lse)
    assert st == 2
    assert "exceeds" in L.mla_last_error()
