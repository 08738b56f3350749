"""Failure detection on the GPU without a fault: every wait in the tensor-core
decode kernel is bounded, and a wait that runs out is reported through the
device error word while the CUDA context stays usable.  The test makes the page
waits run out by having the launch issue no copies (a barrier that nothing
completes), then checks the reported status and that the next call is correct."""
import pytest
import torch

import oracle
from mla_latent_kv_fp8_gb300 import synth
from tests.parity import assert_parity

pytestmark = pytest.mark.gpu

WAIT_TIMEOUT = 1  # device error code of a bounded wait that ran out


@pytest.fixture(scope="module")
def L():
    from mla_latent_kv_fp8_gb300 import build
    build.build()
    from mla_latent_kv_fp8_gb300 import _lib
    _lib.lib()
    return _lib


def _decode(L, case, n_splits):
    B, T, H = case.q.shape[:3]
    out = torch.full((B, T, H, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((B, T, H), float("nan"), dtype=torch.float32, device="cuda")
    L.mla_decode_paged(case.q, case.kv_cache, case.kv_scale, case.block_table, case.seq_lens,
                       n_splits, case.sm_scale, out, lse)
    return out, lse


@pytest.mark.parametrize("lens,H,T,n_splits", [([700, 130], 12, 1, 3), ([300], 32, 2, 0)])
def test_wait_timeout_is_reported_and_context_survives(L, lens, H, T, n_splits):
    case = synth.make_decode_case(31, lens, H, T)
    cg = case.to("cuda")
    prev_impl = L.mla_set_impl(2)  # the tensor-core kernel
    assert L.mla_device_error() == 0
    try:
        L.mla_test_stall_copies(True)
        _decode(L, cg, n_splits)
        torch.cuda.synchronize()  # the launch ends by itself (bounded waits)
        assert L.mla_device_error() == WAIT_TIMEOUT
    finally:
        L.mla_test_stall_copies(False)
        L.mla_set_impl(prev_impl)
    assert L.mla_device_error() == 0  # reading the word cleared it
    # the same context decodes correctly afterwards
    out, lse = _decode(L, cg, n_splits)
    torch.cuda.synchronize()
    assert L.mla_device_error() == 0
    ro, rl = oracle.decode(case.q, case.kv_cache, case.kv_scale, case.block_table, case.seq_lens,
                           case.sm_scale)
    assert_parity(out, lse, ro, rl, what="after a reported timeout")
