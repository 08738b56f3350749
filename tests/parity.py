"""Shared parity criteria for GPU results against the FP64 oracle.

Tolerances (on the bf16 output and the fp32 log-sum-exp):
  max |out - ref|                 <= 1e-2
  max |out - ref| / max |ref|     <= 1.6e-2
  max |lse - lse_ref|             <= 1e-4
Rows whose reference lse is -inf (empty history) must be exactly 0 / -inf.
"""
import numpy as np
import torch

ATOL_OUT = 1e-2
RTOL_OUT = 1.6e-2
ATOL_LSE = 1e-4


def to_np(x):
    if isinstance(x, torch.Tensor):
        return x.detach().float().cpu().numpy().astype(np.float64)
    return np.asarray(x, dtype=np.float64)


def errors(out, lse, ref_out, ref_lse, sel=None):
    o, l = to_np(out), to_np(lse)
    ro, rl = np.asarray(ref_out), np.asarray(ref_lse)
    if sel is not None:
        o, l, ro, rl = o[sel], l[sel], ro[sel], rl[sel]
    empty = np.isneginf(rl)
    res = {"empty_rows": int(empty.sum())}
    if empty.any():
        res["empty_ok"] = bool(np.all(o[empty] == 0) and np.all(np.isneginf(l[empty])))
    full = ~empty
    if full.any():
        d = np.abs(o[full] - ro[full])
        res["max_abs_out"] = float(d.max())
        res["rel_out"] = float(d.max() / max(np.abs(ro[full]).max(), 1e-30))
        res["max_abs_lse"] = float(np.abs(l[full] - rl[full]).max())
        res["norm_rel_out"] = float(np.linalg.norm(o[full] - ro[full]) / np.linalg.norm(ro[full]))
        res["nan"] = bool(np.isnan(o[full]).any() or np.isnan(l[full]).any())
    return res


def assert_parity(out, lse, ref_out, ref_lse, sel=None, what=""):
    e = errors(out, lse, ref_out, ref_lse, sel)
    if "empty_ok" in e:
        assert e["empty_ok"], f"{what}: empty rows must be out=0, lse=-inf: {e}"
    if "max_abs_out" in e:
        assert not e["nan"], f"{what}: NaN in output {e}"
        assert e["max_abs_out"] <= ATOL_OUT, f"{what}: {e}"
        assert e["rel_out"] <= RTOL_OUT, f"{what}: {e}"
        assert e["max_abs_lse"] <= ATOL_LSE, f"{what}: {e}"
    return e
