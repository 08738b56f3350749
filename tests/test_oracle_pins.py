"""Pins for the FP64 oracle: values it must reproduce that do not come from itself.

Each test fixes the oracle against a different external fact: the FP8 format
definition (checked against torch's float8 cast), a 40-digit brute force written
independently here, the invariances the source post states (partition/merge,
head padding), a closed form (constant keys) and two structural reductions
(causal verify = single-token decodes, paging = identity layout).
"""
import json
import math
import os
from decimal import Decimal, getcontext

import numpy as np
import pytest
import torch

import oracle
from mla_latent_kv_fp8_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# --------------------------------------------------------------------------
# FP8 E4M3FN decoding
# --------------------------------------------------------------------------

def test_e4m3fn_all_codes_match_torch_cast(oracle_lib):
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float32).numpy().astype(np.float64)
    got = np.array([oracle_lib.oracle_e4m3fn_to_double(c) for c in range(256)])
    nan_ref = np.isnan(ref)
    assert np.array_equal(nan_ref, np.isnan(got))
    assert nan_ref.sum() == 2 and nan_ref[0x7F] and nan_ref[0xFF]
    assert np.array_equal(ref[~nan_ref], got[~nan_ref])
    assert np.array_equal(np.signbit(ref[~nan_ref]), np.signbit(got[~nan_ref]))


@pytest.mark.parametrize("code,value", [
    (0x7E, 448.0), (0xFE, -448.0), (0x08, 2.0 ** -6), (0x01, 2.0 ** -9), (0x07, 7 * 2.0 ** -9),
    (0x38, 1.0), (0x40, 2.0), (0x3C, 1.5), (0x00, 0.0)])
def test_e4m3fn_format_values(oracle_lib, code, value):
    assert oracle_lib.oracle_e4m3fn_to_double(code) == value


def test_e4m3fn_negative_zero(oracle_lib):
    v = oracle_lib.oracle_e4m3fn_to_double(0x80)
    assert v == 0.0 and math.copysign(1.0, v) == -1.0


# --------------------------------------------------------------------------
# Brute force in 40-digit decimal arithmetic
# --------------------------------------------------------------------------

def _bruteforce(case, rows):
    """Textbook two-pass softmax in Decimal for the listed (b, t, h) rows.

    Written independently of the oracle: codes are decoded with torch's float8
    cast, and every product, exponential and logarithm is taken in 40 digits."""
    getcontext().prec = 40
    kv = case.kv_cache.view(torch.float8_e4m3fn).to(torch.float32).numpy()
    q = case.q.to(torch.float32).numpy()
    bt = case.block_table.numpy()
    lens = case.seq_lens.numpy()
    scale = Decimal(float(case.kv_scale[0]))
    sm = Decimal(case.sm_scale)
    T = case.T
    res = {}
    for (b, t, h) in rows:
        n = int(lens[b]) - T + 1 + t
        qv = [Decimal(float(v)) for v in q[b, t, h]]
        xs, ss = [], []
        for p in range(n):
            row = kv[bt[b, p // 64], p % 64]
            x = [Decimal(float(v)) * scale for v in row]
            xs.append(x)
            ss.append(sm * sum(a * c for a, c in zip(qv, x)))
        m = max(ss)
        w = [(s - m).exp() for s in ss]
        z = sum(w)
        out = [sum(w[i] * xs[i][d] for i in range(n)) / z for d in range(512)]
        res[(b, t, h)] = (np.array([float(v) for v in out]), float(m + z.ln()))
    return res


@pytest.mark.parametrize("T,lens", [(1, [130]), (3, [131, 70])])
def test_oracle_matches_decimal_bruteforce(T, lens):
    case = synth.make_decode_case(101 + T, lens, 2, T, extra_pages=2)
    out, lse = oracle.decode(case.q, case.kv_cache, case.kv_scale, case.block_table,
                             case.seq_lens, case.sm_scale)
    rows = [(b, t, h) for b in range(len(lens)) for t in range(T) for h in range(2)]
    if T > 1:
        rows = rows[::3]
    ref = _bruteforce(case, rows)
    for key, (o_ref, l_ref) in ref.items():
        b, t, h = key
        scale = np.abs(o_ref).max()
        assert np.abs(out[b, t, h] - o_ref).max() <= 1e-12 * scale, key
        assert abs(lse[b, t, h] - l_ref) <= 1e-12 * max(1.0, abs(l_ref)), key


# --------------------------------------------------------------------------
# Partition / merge invariance (post, section 1 DCP and section 4 partitions)
# --------------------------------------------------------------------------

def _partition_masks(kind, n_parts, L, rng):
    if kind == "contiguous":
        cuts = np.sort(rng.choice(np.arange(1, L), size=n_parts - 1, replace=False))
        lab = np.searchsorted(cuts, np.arange(L), side="right")
    elif kind == "interleaved":
        lab = np.arange(L) % n_parts
    elif kind == "random":
        lab = rng.integers(0, n_parts, size=L)
    elif kind == "with_empty":
        lab = rng.integers(0, max(1, n_parts - 2), size=L)  # last two parts stay empty
    else:
        raise ValueError(kind)
    return [(lab == s).astype(np.uint8) for s in range(n_parts)]


@pytest.mark.parametrize("kind", ["contiguous", "interleaved", "random", "with_empty"])
@pytest.mark.parametrize("n_parts", [2, 5, 32])
def test_merge_of_any_partition_equals_whole(kind, n_parts):
    rng = np.random.default_rng([n_parts, len(kind)])
    lens = [300, 211]
    case = synth.make_decode_case(7, lens, 3, 2)
    whole_o, whole_l = oracle.decode(case.q, case.kv_cache, case.kv_scale, case.block_table,
                                     case.seq_lens, case.sm_scale)
    parts_o, parts_l = [], []
    for m in _partition_masks(kind, n_parts, max(lens), rng):
        o, l = oracle.decode(case.q, case.kv_cache, case.kv_scale, case.block_table,
                             case.seq_lens, case.sm_scale, pos_mask=m)
        parts_o.append(o)
        parts_l.append(l)
    mo, ml = oracle.merge(np.stack(parts_o), np.stack(parts_l))
    assert np.abs(mo - whole_o).max() <= 1e-12 * np.abs(whole_o).max()
    assert np.abs(ml - whole_l).max() <= 1e-12 * np.abs(whole_l).max()


def test_merge_all_empty_and_single_part():
    po = np.random.default_rng(0).standard_normal((3, 4, 8))
    pl = np.full((3, 4), -np.inf)
    o, l = oracle.merge(po, pl)
    assert np.all(o == 0) and np.all(np.isneginf(l))
    pl1 = np.array([[0.5, -1.0, 2.0, 3.0]])
    o1, l1 = oracle.merge(po[:1], pl1)
    assert np.array_equal(l1, pl1[0]) and np.allclose(o1, po[0], rtol=0, atol=1e-15)


def test_merge_two_parts_closed_form():
    # two parts with lse a, b: weights e^a/(e^a+e^b), e^b/(e^a+e^b)
    a, b = 1.25, -0.5
    po = np.stack([np.full((1, 4), 2.0), np.full((1, 4), -1.0)])
    o, l = oracle.merge(po, np.array([[a], [b]]))
    wa = 1.0 / (1.0 + math.exp(b - a))
    assert abs(l[0] - (a + math.log1p(math.exp(b - a)))) < 1e-15
    assert np.allclose(o, 2.0 * wa - 1.0 * (1 - wa), rtol=0, atol=1e-15)


# --------------------------------------------------------------------------
# Head padding (post, section 4: padding 12 heads to 16 by copying 4)
# --------------------------------------------------------------------------

def test_head_padding_leaves_original_heads_bit_identical():
    case = synth.make_decode_case(12, [333, 90], 12, 1)
    o12, l12 = oracle.decode(case.q, case.kv_cache, case.kv_scale, case.block_table,
                             case.seq_lens, case.sm_scale)
    q16 = torch.cat([case.q, case.q[:, :, 0:4]], dim=2)
    o16, l16 = oracle.decode(q16, case.kv_cache, case.kv_scale, case.block_table,
                             case.seq_lens, case.sm_scale)
    assert np.array_equal(o16[:, :, :12], o12) and np.array_equal(l16[:, :, :12], l12)
    assert np.array_equal(o16[:, :, 12:], o12[:, :, 0:4])


# --------------------------------------------------------------------------
# Closed form: constant keys give the mean of the values
# --------------------------------------------------------------------------

@pytest.mark.parametrize("zero_q", [False, True])
def test_constant_key_closed_form(zero_q):
    L = 200
    case = synth.make_decode_case(21, [L], 4, 1)
    kv = case.kv_cache.clone()
    bt = case.block_table.numpy()
    # every position shares the same positional bytes [512:576)
    ref_rope = kv[bt[0, 0], 0, 512:].clone()
    for p in range(L):
        kv[bt[0, p // 64], p % 64, 512:] = ref_rope
    q = case.q.clone()
    q[..., :512] = 0
    if zero_q:
        q.zero_()
    o, l = oracle.decode(q, kv, case.kv_scale, case.block_table, case.seq_lens, case.sm_scale)
    xs = kv.view(torch.float8_e4m3fn).to(torch.float32).numpy().astype(np.float64)
    scale = float(case.kv_scale[0])
    rows = np.stack([xs[bt[0, p // 64], p % 64] for p in range(L)]) * scale
    mean = rows[:, :512].mean(axis=0)
    for h in range(4):
        s0 = case.sm_scale * float(np.dot(q[0, 0, h].to(torch.float32).numpy().astype(np.float64),
                                          rows[0]))
        assert np.abs(o[0, 0, h] - mean).max() <= 1e-12 * np.abs(mean).max()
        assert abs(l[0, 0, h] - (s0 + math.log(L))) <= 1e-12 * max(1, abs(s0 + math.log(L)))
        if zero_q:
            assert abs(l[0, 0, h] - math.log(L)) <= 1e-13


# --------------------------------------------------------------------------
# Causal verify reduces to single-token decodes; paging is invisible
# --------------------------------------------------------------------------

def test_causal_verify_equals_single_token_decodes():
    lens = [260, 129]
    case = synth.make_decode_case(31, lens, 3, 4)
    o4, l4 = oracle.decode(case.q, case.kv_cache, case.kv_scale, case.block_table,
                           case.seq_lens, case.sm_scale)
    for t in range(4):
        sl = case.seq_lens - 3 + t
        o1, l1 = oracle.decode(case.q[:, t:t + 1].contiguous(), case.kv_cache, case.kv_scale,
                               case.block_table, sl, case.sm_scale)
        assert np.array_equal(o1[:, 0], o4[:, t]) and np.array_equal(l1[:, 0], l4[:, t])
    # the causal rule is not vacuous: rows t differ
    assert not np.array_equal(l4[:, 0], l4[:, 3])


def test_dcp_verify_decomposition_equals_unsharded():
    """Multi-token verify over a history cut into contiguous DCP shards (post,
    section 1): every shard but the last holds only positions that all T draft
    queries see, so it is a T = 1 decode of T*H independent rows; the last shard
    holds the T draft positions and keeps the causal rule.  Merging the shards'
    (out, lse) equals the unsharded causal verify."""
    T, H, n = 4, 3, 4
    sc = synth.make_sharded_case(17, 2, H, 4 * 96, n, T=T)
    outs, lses = [], []
    for s, sh in enumerate(sc.shards):
        B = sh.q.shape[0]
        if s < n - 1:
            q1 = sh.q.reshape(B, 1, T * H, 576).contiguous()
            o, l = oracle.decode(q1, sh.kv_cache, sh.kv_scale, sh.block_table, sh.seq_lens, sh.sm_scale)
            o, l = o.reshape(B, T, H, 512), l.reshape(B, T, H)
        else:
            o, l = oracle.decode(sh.q, sh.kv_cache, sh.kv_scale, sh.block_table, sh.seq_lens, sh.sm_scale)
        outs.append(o)
        lses.append(l)
    mo, ml = oracle.merge(np.stack(outs), np.stack(lses))
    ro, rl = oracle.decode(sc.full.q, sc.full.kv_cache, sc.full.kv_scale, sc.full.block_table,
                           sc.full.seq_lens, sc.full.sm_scale)
    np.testing.assert_allclose(mo, ro, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(ml, rl, rtol=1e-12, atol=1e-12)
    # the causal rule inside the last shard matters: treating it as T = 1 differs
    last = sc.shards[-1]
    q1 = last.q.reshape(2, 1, T * H, 576).contiguous()
    _, l_wrong = oracle.decode(q1, last.kv_cache, last.kv_scale, last.block_table, last.seq_lens,
                               last.sm_scale)
    assert not np.allclose(l_wrong.reshape(2, T, H), lses[-1])


def test_permuted_block_table_equals_identity_layout():
    lens = [300, 64, 1]
    case = synth.make_decode_case(41, lens, 2, 1, extra_pages=5)
    bt = case.block_table.numpy()
    pages = [(L + 63) // 64 for L in lens]
    order = [int(bt[b, j]) for b in range(len(lens)) for j in range(pages[b])]
    kv_id = case.kv_cache[torch.tensor(order, dtype=torch.long)].contiguous()
    bt_id = np.zeros_like(bt)
    off = 0
    for b in range(len(lens)):
        bt_id[b, :pages[b]] = np.arange(off, off + pages[b])
        off += pages[b]
    o_p, l_p = oracle.decode(case.q, case.kv_cache, case.kv_scale, case.block_table,
                             case.seq_lens, case.sm_scale)
    o_i, l_i = oracle.decode(case.q, kv_id, case.kv_scale, torch.from_numpy(bt_id),
                             case.seq_lens, case.sm_scale)
    assert np.array_equal(o_p, o_i) and np.array_equal(l_p, l_i)


def test_empty_history_gives_zero_and_neg_inf():
    case = synth.make_decode_case(5, [0, 70], 2, 1)
    o, l = oracle.decode(case.q, case.kv_cache, case.kv_scale, case.block_table,
                         case.seq_lens, case.sm_scale)
    assert np.all(o[0] == 0) and np.all(np.isneginf(l[0]))
    assert np.all(np.isfinite(l[1]))


def test_invalid_inputs_are_rejected():
    case = synth.make_decode_case(5, [3], 2, 1)
    with pytest.raises(ValueError):
        # T=4 new positions but only 3 cached
        oracle.decode(torch.cat([case.q] * 4, dim=1), case.kv_cache, case.kv_scale,
                      case.block_table, case.seq_lens, case.sm_scale)
    bad_bt = case.block_table.clone()
    bad_bt[0, 0] = case.kv_cache.shape[0]
    with pytest.raises(ValueError):
        oracle.decode(case.q, case.kv_cache, case.kv_scale, bad_bt, case.seq_lens, case.sm_scale)


def test_row_mask_computes_only_selected_rows():
    case = synth.make_decode_case(8, [150, 77], 3, 2)
    o, l = oracle.decode(case.q, case.kv_cache, case.kv_scale, case.block_table,
                         case.seq_lens, case.sm_scale)
    rm = np.zeros((2, 2, 3), dtype=np.uint8)
    rm[1, 0, 2] = rm[0, 1, 0] = 1
    o2, l2 = oracle.decode(case.q, case.kv_cache, case.kv_scale, case.block_table,
                           case.seq_lens, case.sm_scale, row_mask=rm)
    sel = rm.astype(bool)
    assert np.array_equal(o2[sel], o[sel]) and np.array_equal(l2[sel], l[sel])


# --------------------------------------------------------------------------
# The post's worked byte count (section 1: 24 x 142,000 x 576 FP8 bytes)
# --------------------------------------------------------------------------

def test_payload_byte_accounting_matches_post():
    with open(os.path.join(GOLDEN, "mla_payload_bytes.json")) as f:
        g = json.load(f)
    total = synth.mla_payload_bytes(g["layers"], g["positions"])
    assert total == g["layers"] * g["positions"] * g["bytes_per_position"]
    assert round(total / 1e9, 2) == g["per_gpu_gb_tp8"]
    assert round(synth.mla_payload_bytes(g["layers"], g["positions"], g["dcp"]) / 1e6) == \
        g["per_gpu_mb_dcp8"]
    case = synth.make_decode_case(1, [100, 37], 2, 1)
    assert case.kv_bytes() == 137 * 576


# --------------------------------------------------------------------------
# Latent append: E4M3FN encoding and the paged write
# --------------------------------------------------------------------------

def _torch_encode(x32):
    """Independent quantiser: torch's float8_e4m3fn cast (round to nearest even)
    after clamping to the largest finite magnitude."""
    return torch.clamp(torch.as_tensor(x32, dtype=torch.float32), -448.0, 448.0).to(
        torch.float8_e4m3fn).view(torch.uint8).numpy()


@pytest.mark.parametrize("scale", [1.0, 0.0091, 2.0 ** -5, 3.7])
def test_e4m3fn_encode_matches_torch_cast(scale):
    bits = np.arange(1 << 16, dtype=np.uint32) << 16
    x = bits.view(np.float32)
    x = x[np.isfinite(x)]
    v = (x / np.float32(scale)).astype(np.float32)  # binary32 division, as the append does
    assert np.array_equal(oracle.e4m3fn_encode(v), _torch_encode(v))


def test_e4m3fn_encode_random_binary32_matches_torch_cast():
    rng = np.random.default_rng(5)
    v = (rng.standard_normal(200000) * np.exp(rng.uniform(-12, 7, 200000))).astype(np.float32)
    assert np.array_equal(oracle.e4m3fn_encode(v), _torch_encode(v))


def test_e4m3fn_encode_round_trips_every_finite_code():
    codes = [c for c in range(256) if c not in (0x7F, 0xFF)]
    vals = np.array([oracle.e4m3fn_to_double(c) for c in codes], dtype=np.float32)
    assert list(oracle.e4m3fn_encode(vals)) == codes


@pytest.mark.parametrize("x,code", [
    (1.0625, 0x38),        # tie between 1 and 1.125: even mantissa (1.0)
    (17.0, 0x58),          # tie between 16 and 18 -> 16
    (19.0, 0x5A),          # tie between 18 and 20 -> 20
    (2.0 ** -10, 0x00),    # tie between 0 and the smallest subnormal -> 0
    (1.5 * 2.0 ** -9, 0x02),
    (-2.0 ** -11, 0x80),   # rounds to -0
    (448.0, 0x7E), (464.0, 0x7E), (1e30, 0x7E), (-1e30, 0xFE),  # saturation
])
def test_e4m3fn_encode_ties_and_saturation(x, code):
    assert int(oracle.e4m3fn_encode(np.array([x], dtype=np.float32))[0]) == code


def _append_case(lib=None):
    """(new cache from the oracle, cache expected from torch's quantiser, old cache)."""
    rng = np.random.default_rng(9)
    num_pages, B, T = 12, 3, 3
    kv = rng.integers(0, 0x7E, size=(num_pages, 64, 576), dtype=np.uint8)
    bt = rng.permutation(num_pages)[:B * 4].reshape(B, 4).astype(np.int32)
    start = np.array([62, 0, 190], dtype=np.int32)  # crosses a page boundary; the last page
    lat = torch.from_numpy(rng.standard_normal((B, T, 576)).astype(np.float32) * 3).to(torch.bfloat16)
    lat[0, 1, 7] = 5000.0  # saturates
    scale = np.float32(0.0123)
    new, rc = oracle.append_latent(lat, torch.tensor([scale]), bt, start, kv, lib=lib)
    assert rc == 0
    expect = kv.copy()
    for b in range(B):
        for t in range(T):
            p = int(start[b]) + t
            v = (lat[b, t].float().numpy() / scale).astype(np.float32)
            expect[bt[b, p // 64], p % 64] = _torch_encode(v)
    return new, expect, kv


def test_append_writes_exactly_the_new_rows():
    new, expect, old = _append_case()
    assert np.array_equal(new, expect)
    assert not np.array_equal(new, old)


def test_append_skips_rows_out_of_range():
    num_pages = 4
    kv = np.zeros((num_pages, 64, 576), dtype=np.uint8)
    bt = np.array([[0, 1], [2, 9]], dtype=np.int32)  # request 1's second page id is out of range
    lat = torch.ones((2, 2, 576), dtype=torch.bfloat16)
    new, rc = oracle.append_latent(lat, torch.tensor([1.0]), bt, np.array([127, 63], dtype=np.int32), kv)
    assert rc == -2
    assert (new[1, 63] == 0x38).all()           # request 0, position 127: written
    assert (new[2, 63] == 0x38).all()           # request 1, position 63: written
    assert int(new.astype(np.int64).sum()) == 2 * 576 * 0x38   # positions 128 / 64 (bad page): skipped
