"""The oracle's pins must be sensitive: plant plausible mistakes in a temporary
copy of the oracle source (a dropped term, a wrong index, a wrong sign or
offset, a misplaced scale) and check that at least one pin fails for each.
The planted copies are compiled into a temporary directory; the committed
oracle is never modified."""
import math
import os
import subprocess

import numpy as np
import pytest
import torch

import oracle
from mla_latent_kv_fp8_gb300 import synth
from tests.test_oracle_pins import _append_case, _bruteforce, _torch_encode

SRC = os.path.join(os.path.dirname(oracle.__file__), "mla_oracle.c")

MUTANTS = {
    "drop_positional_dims": ("for (int d = 0; d < ORACLE_DQK; ++d)\n                acc +=",
                             "for (int d = 0; d < ORACLE_DV; ++d)\n                acc +="),
    "value_from_wrong_dims": ("x[d] = J->lut[codes[d]];\n        for (int h = 0; h < H; ++h) {\n            if (!row_wanted(J, b, t, h))\n                continue;\n            double w",
                              "x[d] = J->lut[codes[d + 64]];\n        for (int h = 0; h < H; ++h) {\n            if (!row_wanted(J, b, t, h))\n                continue;\n            double w"),
    "causal_off_by_one": ("L - J->T + 1 + t;", "L - J->T + t;"),
    "page_row_index": ("p % ORACLE_PAGE) * ORACLE_DQK", "(p + 1) % ORACLE_PAGE) * ORACLE_DQK"),
    "lse_missing_max": ("mx[h] + log(z[h]);", "log(z[h]);"),
    "scale_missing": ("oracle_e4m3fn_to_double((uint8_t)c) * J->kv_scale;",
                      "oracle_e4m3fn_to_double((uint8_t)c);"),
    "exponent_bias": ("ldexp(1.0 + (double)m / 8.0, e - 7)", "ldexp(1.0 + (double)m / 8.0, e - 8)"),
    "merge_weight_uses_max": ("double w = exp(ls - total);", "double w = exp(ls - m);"),
    "sm_scale_dropped": ("score[(int64_t)h * n + cnt] = J->sm_scale * acc;",
                         "score[(int64_t)h * n + cnt] = acc;"),
    "block_table_row": ("J->block_table[(int64_t)b * J->bt_stride + p / ORACLE_PAGE]",
                        "J->block_table[(int64_t)b + (p / ORACLE_PAGE) * J->bt_stride]"),
    "encode_tie_away_from_even": ("pick = (c & 1) == 0 ? c : c + 1;", "pick = c + 1;"),
    "encode_overflow_to_nan": ("if (a >= 448.0)\n        return sign | 0x7E;",
                               "if (a >= 448.0)\n        return sign | 0x7F;"),
    "append_row_index": ("kv + ((int64_t)page * ORACLE_PAGE + p % ORACLE_PAGE) * ORACLE_DQK;",
                         "kv + ((int64_t)page * ORACLE_PAGE + (p + 1) % ORACLE_PAGE) * ORACLE_DQK;"),
    "append_scale_multiplies": ("float v = f / kv_scale;", "float v = f * kv_scale;"),
    "lse_in_log2": ("mx[h] + log(z[h]);", "mx[h] + log2(z[h]);"),
    "output_not_normalised": ("o[d] /= z[h];", "o[d] = o[d];"),
    "merge_lse_missing_max": ("double total = m + log(sum);", "double total = log(sum);"),
    "subnormal_exponent": ("ldexp((double)m / 8.0, 1 - 7)", "ldexp((double)m / 8.0, -7)"),
    "mantissa_width": ("ldexp(1.0 + (double)m / 8.0, e - 7)", "ldexp(1.0 + (double)m / 16.0, e - 7)"),
    "causal_ignored": ("L - J->T + 1 + t;", "L;"),
}


def _pins_pass(lib):
    """A compact battery of the external pins; False as soon as one fails
    (an oracle that rejects valid inputs fails too)."""
    try:
        return _battery(lib)
    except ValueError:
        return False


def _battery(lib):
    # FP8 format vs torch's cast
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).float().numpy()
    got = np.array([lib.oracle_e4m3fn_to_double(c) for c in range(256)], dtype=np.float32)
    fin = np.isfinite(ref)
    if not np.array_equal(ref[fin], got[fin]):
        return False
    # decimal brute force, single token and causal verify, permuted pages
    for T, lens in [(1, [130, 70]), (3, [131])]:
        case = synth.make_decode_case(101 + T, lens, 2, T, extra_pages=2)
        out, lse = oracle.decode(case.q, case.kv_cache, case.kv_scale, case.block_table,
                                 case.seq_lens, case.sm_scale, lib=lib)
        rows = [(b, t, h) for b in range(len(lens)) for t in range(T) for h in range(2)][::2]
        for (b, t, h), (o_ref, l_ref) in _bruteforce(case, rows).items():
            if np.abs(out[b, t, h] - o_ref).max() > 1e-12 * np.abs(o_ref).max():
                return False
            if abs(lse[b, t, h] - l_ref) > 1e-12 * max(1.0, abs(l_ref)):
                return False
    # merge of a contiguous partition equals the whole
    case = synth.make_decode_case(7, [300], 2, 1)
    wo, wl = oracle.decode(case.q, case.kv_cache, case.kv_scale, case.block_table,
                           case.seq_lens, case.sm_scale, lib=lib)
    parts = [np.r_[np.ones(100), np.zeros(200)], np.r_[np.zeros(100), np.ones(200)]]
    po, pl = zip(*[oracle.decode(case.q, case.kv_cache, case.kv_scale, case.block_table,
                                 case.seq_lens, case.sm_scale, pos_mask=m.astype(np.uint8), lib=lib)
                   for m in parts])
    mo, ml = oracle.merge(np.stack(po), np.stack(pl), lib=lib)
    if np.abs(mo - wo).max() > 1e-12 * np.abs(wo).max() or np.abs(ml - wl).max() > 1e-12 * np.abs(wl).max():
        return False
    # E4M3FN encoding vs torch's quantiser, and the placement of appended rows
    rng = np.random.default_rng(3)
    v = np.r_[rng.standard_normal(4000) * np.exp(rng.uniform(-12, 7, 4000)),
              np.linspace(440, 500, 121), [17.0, 19.0, 1.0625, 2.0 ** -10]].astype(np.float32)
    if not np.array_equal(oracle.e4m3fn_encode(v, lib=lib), _torch_encode(v)):
        return False
    new, expect, _ = _append_case(lib)
    return bool(np.array_equal(new, expect))


@pytest.fixture(scope="module")
def mutant_dir(tmp_path_factory):
    return tmp_path_factory.mktemp("oracle_mutants")


def test_unmodified_oracle_passes_battery():
    assert _pins_pass(oracle.load())


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name, mutant_dir):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation target for {name} not found in the oracle source"
    path_c = os.path.join(mutant_dir, f"{name}.c")
    path_so = os.path.join(mutant_dir, f"lib{name}.so")
    with open(path_c, "w") as f:
        f.write(src.replace(old, new, 1))
    subprocess.run(["gcc", "-O2", "-std=gnu11", "-ffp-contract=off", "-fPIC", "-shared", "-pthread",
                    "-o", path_so, path_c, "-lm"], check=True)
    lib = oracle.load(path_so)
    assert not _pins_pass(lib), f"pins did not detect the planted mistake '{name}'"
