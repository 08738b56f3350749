"""The cross-GPU DCP exchange (mla_latent_kv_fp8_gb300.dcp) on CPU ranks (gloo,
world sizes 2 and 3): section 1 "Cache", DCP paragraph of the post -- every rank holds
one contiguous shard of every history; the queries are all-gathered so every
rank attends with all heads to its shard; the partial answers (out, lse) are
all-gathered and merged by their normalisers.

The product's exchange and bookkeeping run as they would on GPUs; only the two
compute steps are replaced by data: each rank's local partial answer is
precomputed by the FP64 oracle on its shard (as the decode kernel would
produce it), and the merge is an oracle merge on the test side.  The test
checks that the gathered queries are every rank's heads in rank order, that
the gathered partials are every shard's answer in rank order, and that the
merged answer of each rank's heads equals the unsharded oracle."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle
from mla_latent_kv_fp8_gb300 import dcp, synth


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _shard_partials(case, plan, T):
    """The oracle's answer of every shard over all heads: a shard before the last
    as T = 1 with T*H rows (all its positions precede every draft query), the
    last one with the causal rule."""
    B, H = case.B, case.H
    parts = []
    for s, (bt, sl) in enumerate(plan):
        if s < len(plan) - 1 and T > 1:
            o, l = oracle.decode(case.q.reshape(B, 1, T * H, 576), case.kv_cache, case.kv_scale, bt, sl,
                                 case.sm_scale)
            o, l = o.reshape(B, T, H, 512), l.reshape(B, T, H)
        else:
            o, l = oracle.decode(case.q, case.kv_cache, case.kv_scale, bt, sl, case.sm_scale)
        parts.append((o, l))
    return parts


def _rank_main(rank, world, port, q_full, partials, dtype, result):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        H = q_full.shape[2]
        Hl = H // world
        q_local = q_full[:, :, rank * Hl:(rank + 1) * Hl].clone()
        seen = {}

        def local_decode(q_all):
            seen["q_all"] = q_all.clone()
            o, l = partials[rank]
            return torch.from_numpy(o).to(dtype), torch.from_numpy(l).float()

        def merge(po, pl):
            seen["po"], seen["pl"] = po.clone(), pl.clone()
            o, l = oracle.merge(po.double().numpy(), pl.double().numpy())
            return torch.from_numpy(o), torch.from_numpy(l)

        out, lse, _ = dcp.dcp_decode(q_local, local_decode, merge)
        result[rank] = (out.numpy(), lse.numpy(), seen["q_all"].float().numpy(), seen["po"].float().numpy(),
                        seen["pl"].numpy())
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world,T,dtype", [(2, 1, torch.float64), (2, 4, torch.float64), (2, 4, torch.bfloat16),
                                           (3, 4, torch.float64)])
def test_dcp_exchange_matches_unsharded_oracle(world, T, dtype):
    H = 12
    lens = [1500, 700, 900]
    case = synth.make_decode_case(41 + T, lens, H, T, extra_pages=3)
    plan = dcp.shard_plan(lens, case.block_table, world, T)
    partials = _shard_partials(case, plan, T)
    ro, rl = oracle.decode(case.q, case.kv_cache, case.kv_scale, case.block_table, case.seq_lens, case.sm_scale)

    port = _free_port()
    result = mp.get_context("spawn").Manager().dict()
    mp.spawn(_rank_main, args=(world, port, case.q, partials, dtype, result), nprocs=world, join=True)

    Hl = H // world
    for r in range(world):
        out, lse, q_all, po, pl = result[r]
        # every rank gathered all heads, rank r's at [r * Hl, (r + 1) * Hl)
        assert np.array_equal(q_all, case.q.float().numpy())
        # and every shard's partial answer, in rank order
        for s in range(world):
            ref_o = torch.from_numpy(partials[s][0]).to(dtype).float().numpy()
            assert np.array_equal(po[s], ref_o)
            assert np.array_equal(pl[s], partials[s][1].astype(np.float32))
        sl = slice(r * Hl, (r + 1) * Hl)
        if dtype == torch.float64:
            # exact bookkeeping: the merge of the shards is the unsharded answer
            # (up to the fp32 transport of the LSEs)
            np.testing.assert_allclose(out, ro[:, :, sl], atol=1e-6, rtol=0)
            np.testing.assert_allclose(lse, rl[:, :, sl], atol=1e-5, rtol=0)
        else:
            from tests.parity import assert_parity
            assert_parity(torch.from_numpy(out), torch.from_numpy(lse), ro[:, :, sl], rl[:, :, sl],
                          what=f"DCP exchange, rank {r}, bf16 partials")


def test_shard_plan_tiles_each_history_in_order():
    lens = synth.verify_lens(4)
    B, T = len(lens), 4
    mp_ = -(-max(lens) // 64)
    bt = torch.stack([torch.randperm(10 * mp_)[:mp_] for _ in range(B)]).to(torch.int32)
    for n in (2, 8):
        plan = dcp.shard_plan(lens, bt, n, T)
        for b, L in enumerate(lens):
            pages, pos = [], 0
            for s, (table, sl) in enumerate(plan):
                k = int(sl[b])
                if s < n - 1:
                    assert k % 64 == 0
                pages += table[b, :-(-k // 64)].tolist()
                pos += k
            assert pos == L and pages == bt[b, :-(-L // 64)].tolist()
            assert int(plan[-1][1][b]) >= T
