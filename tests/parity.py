"""Shared parity criteria for GPU results against the FP64 oracle.

Tolerances (on the bf16 output and the fp32 log-sum-exp), element by element:
  |out - ref|                     <= 1e-2 + ulp_bf16(ref) / 2
  max |out - ref| / max |ref|     <= 1.6e-2
  |lse - lse_ref|                 <= max(1e-4, 2^-20 |lse_ref|)
The output is bf16, so the exact answer itself, rounded to bf16, is off by up
to half a bf16 ulp: the absolute bound is read on top of that rounding (which
exceeds 1e-2 on its own wherever |ref| >= 4).  The LSE bound is absolute for
log-sum-exps up to ~105 and relative (2^-20, about 8 fp32 ulps) beyond, where
fp32 itself cannot hold 1e-4 (its ulp reaches 1e-4 at |lse| = 1,024).
Rows whose reference lse is -inf (empty history) must be exactly 0 / -inf.
"""
import numpy as np
import torch

ATOL_OUT = 1e-2
RTOL_OUT = 1.6e-2
ATOL_LSE = 1e-4
RTOL_LSE = 2.0 ** -20


def to_np(x):
    if isinstance(x, torch.Tensor):
        return x.detach().float().cpu().numpy().astype(np.float64)
    return np.asarray(x, dtype=np.float64)


def bf16_half_ulp(ref):
    """Half the spacing of bf16 values at |ref| (8 significant bits)."""
    a = np.abs(np.asarray(ref, dtype=np.float64))
    _, e = np.frexp(np.maximum(a, 2.0 ** -126))  # a = m * 2^e, m in [0.5, 1)
    return np.ldexp(1.0, e - 9)


def out_bound(ref):
    return ATOL_OUT + bf16_half_ulp(ref)


def lse_bound(ref):
    return np.maximum(ATOL_LSE, RTOL_LSE * np.abs(np.asarray(ref, dtype=np.float64)))


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
        dl = np.abs(l[full] - rl[full])
        res["max_abs_out"] = float(d.max())
        res["out_bound_used"] = float((d / out_bound(ro[full])).max())  # <= 1 passes
        res["rel_out"] = float(d.max() / max(np.abs(ro[full]).max(), 1e-30))
        res["max_abs_lse"] = float(dl.max())
        res["lse_bound_used"] = float((dl / lse_bound(rl[full])).max())  # <= 1 passes
        res["norm_rel_out"] = float(np.linalg.norm(o[full] - ro[full]) / np.linalg.norm(ro[full]))
        res["nan"] = bool(np.isnan(o[full]).any() or np.isnan(l[full]).any())
    return res


def assert_parity(out, lse, ref_out, ref_lse, sel=None, what=""):
    e = errors(out, lse, ref_out, ref_lse, sel)
    if "empty_ok" in e:
        assert e["empty_ok"], f"{what}: empty rows must be out=0, lse=-inf: {e}"
    if "max_abs_out" in e:
        assert not e["nan"], f"{what}: NaN in output {e}"
        assert e["out_bound_used"] <= 1.0, f"{what}: {e}"
        assert e["rel_out"] <= RTOL_OUT, f"{what}: {e}"
        assert e["lse_bound_used"] <= 1.0, f"{what}: {e}"
    return e
