"""GPU parity of mla_append_latent (the latent-cache append before each decode
step) against the oracle: the whole cache must be byte-identical after the
append, and a decode over the appended cache must match the oracle's decode of
the oracle-appended cache."""
import numpy as np
import pytest
import torch

import oracle
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


def _append_both(L, case, latent, start):
    """Append on the GPU (in a copy of the cache) and in the oracle; return both caches."""
    kv_gpu = case.kv_cache.clone().cuda()
    st = torch.tensor(start, dtype=torch.int32)
    L.mla_append_latent(latent.cuda(), case.kv_scale.cuda(), case.block_table.cuda(), st.cuda(), kv_gpu)
    torch.cuda.synchronize()
    err = L.mla_device_error()
    kv_ref, rc = oracle.append_latent(latent, case.kv_scale, case.block_table, st, case.kv_cache.cpu())
    return kv_gpu.cpu().numpy(), kv_ref, err, rc


@pytest.mark.parametrize("lens,T,amp", [
    ([64, 1, 200, 129, 700], 1, 1.0),
    ([66, 130, 4, 1000], 4, 3.0),      # positions cross page boundaries
    ([63, 128], 2, 1000.0),            # most values saturate at +-448
])
def test_append_is_byte_identical_to_oracle(L, lens, T, amp):
    case = synth.make_decode_case(300 + T, lens, 12, T, extra_pages=2)
    latent = synth.make_latent(400 + T, len(lens), T, amplitude=amp)
    start = [x - T for x in lens]
    got, ref, err, rc = _append_both(L, case, latent, start)
    assert err == 0 and rc == 0
    assert np.array_equal(got, ref)


def test_append_then_decode_matches_oracle(L):
    lens, T = [517, 64, 3000], 4
    case = synth.make_decode_case(501, lens, 12, T, extra_pages=1)
    # same distribution as the history: outputs stay weighted averages of |x| < ~4,
    # where bf16 rounding (half an ulp) stays under the 1e-2 absolute bound
    latent = synth.make_latent(502, len(lens), T, amplitude=1.0)
    start = [x - T for x in lens]
    kv_gpu = case.kv_cache.clone().cuda()
    g = case.to("cuda")
    L.mla_append_latent(latent.cuda(), g.kv_scale, g.block_table,
                        torch.tensor(start, dtype=torch.int32, device="cuda"), kv_gpu)
    out = torch.full((len(lens), T, 12, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((len(lens), T, 12), float("nan"), device="cuda")
    L.mla_decode_paged(g.q, kv_gpu, g.kv_scale, g.block_table, g.seq_lens, 0, g.sm_scale, out, lse)
    torch.cuda.synchronize()
    assert L.mla_device_error() == 0
    kv_ref, rc = oracle.append_latent(latent, case.kv_scale, case.block_table, torch.tensor(start), case.kv_cache)
    assert rc == 0 and np.array_equal(kv_gpu.cpu().numpy(), kv_ref)
    ro, rl = oracle.decode(case.q, kv_ref, case.kv_scale, case.block_table, case.seq_lens, case.sm_scale)
    assert_parity(out, lse, ro, rl, what="decode after append")


def test_append_out_of_range_rows_are_skipped_and_reported(L):
    case = synth.make_decode_case(601, [128, 128], 12, 1)
    latent = synth.make_latent(602, 2, 2)
    # request 0 would write positions 127, 128 (the second is past the block table);
    # request 1 writes 0, 1 normally
    got, ref, err, rc = _append_both(L, case, latent, [127, 0])
    assert rc == -2 and err == 3          # a position out of range was skipped
    assert np.array_equal(got, ref)
    bt = case.block_table.clone()
    bt[1, 0] = 10_000                      # request 1's first page id is out of range
    case.block_table = bt
    got, ref, err, rc = _append_both(L, case, latent, [0, 0])
    assert rc == -2 and err == 2
    assert np.array_equal(got, ref)


def test_full_size_append_tp8_and_verify_shapes(L):
    for name, T in (("tp8_batch", 1), ("verify", 4)):
        case = synth.workload_case(name, device="cuda")
        B = case.q.shape[0]
        latent = synth.make_latent(700 + T, B, T, amplitude=1.0)
        start = [x - T for x in case.lens]
        kv_gpu = case.kv_cache.clone()
        L.mla_append_latent(latent.cuda(), case.kv_scale, case.block_table,
                            torch.tensor(start, dtype=torch.int32, device="cuda"), kv_gpu)
        torch.cuda.synchronize()
        assert L.mla_device_error() == 0
        # compare only the written rows (the oracle would copy the whole multi-GB pool)
        bt = case.block_table.cpu().numpy()
        for b in range(B):
            for t in range(T):
                p = start[b] + t
                row = kv_gpu[bt[b, p // 64], p % 64].cpu().numpy()
                v = (latent[b, t].float().numpy() / np.float32(case.kv_scale.item())).astype(np.float32)
                assert np.array_equal(row, oracle.e4m3fn_encode(v)), (name, b, t)
        del kv_gpu, case
