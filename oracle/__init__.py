"""FP64 CPU oracle for paged FP8 latent-KV MLA decode and the LSE merge.

TEST INFRASTRUCTURE ONLY.  Only the test suite, ``__graft_entry__.smoke()`` and
the benchmark's CPU-baseline leg may import this package.  The product path
(``mla_latent_kv_fp8_gb300``) never imports it and shares no code with it.

The arithmetic lives in ``mla_oracle.c`` (plain C, double precision); this
module compiles it with gcc on first use and marshals numpy/torch arrays.
Every function states the definition it computes; see the C file for the
passages of the source post each step follows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mla_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libmla_oracle.so")
_lock = threading.Lock()
_lib = None

PAGE = 64
D_QK = 576
D_V = 512


def build(force: bool = False, defines: tuple[str, ...] = (), out_path: str | None = None) -> str:
    """Compile the oracle shared library with gcc (strict IEEE, no FMA contraction)."""
    out_path = out_path or _LIB_PATH
    if (not force and not defines and os.path.exists(out_path)
            and os.path.getmtime(out_path) >= os.path.getmtime(_SRC)):
        return out_path
    tmp = out_path + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=gnu11", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
           "-shared", "-pthread", *[f"-D{d}" for d in defines], "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out_path)
    return out_path


def load(path: str | None = None):
    """Load (building if needed) the oracle library and declare its signatures."""
    global _lib
    with _lock:
        if path is None and _lib is not None:
            return _lib
        lib = ctypes.CDLL(path or build())
        P = ctypes.c_void_p
        lib.oracle_e4m3fn_to_double.argtypes = [ctypes.c_uint8]
        lib.oracle_e4m3fn_to_double.restype = ctypes.c_double
        lib.oracle_mla_decode.argtypes = [
            P, P, ctypes.c_int64, ctypes.c_float, P, ctypes.c_int64, P,
            ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_double,
            P, ctypes.c_int64, P, P, P, ctypes.c_int]
        lib.oracle_mla_decode.restype = ctypes.c_int
        lib.oracle_lse_merge.argtypes = [ctypes.c_int, ctypes.c_int64, ctypes.c_int, P, P, P, P]
        lib.oracle_lse_merge.restype = ctypes.c_int
        lib.oracle_e4m3fn_encode.argtypes = [ctypes.c_float]
        lib.oracle_e4m3fn_encode.restype = ctypes.c_uint8
        lib.oracle_e4m3fn_encode_array.argtypes = [P, ctypes.c_int64, P]
        lib.oracle_e4m3fn_encode_array.restype = None
        lib.oracle_append_latent.argtypes = [P, ctypes.c_int, ctypes.c_int, ctypes.c_float, P,
                                             ctypes.c_int64, ctypes.c_int, P, P, ctypes.c_int64]
        lib.oracle_append_latent.restype = ctypes.c_int
        if path is None:
            _lib = lib
        return lib


def _np(x, dtype):
    """torch tensor or array-like -> C-contiguous numpy array of ``dtype`` (no value change)."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().cpu()
            if x.dtype == torch.bfloat16:
                x = x.view(torch.int16)
            elif x.dtype == torch.float8_e4m3fn:
                x = x.view(torch.uint8)
            x = x.contiguous().numpy()
    except ImportError:  # pragma: no cover
        pass
    a = np.asarray(x)
    if a.dtype != dtype:
        if a.dtype.itemsize == np.dtype(dtype).itemsize and a.dtype.kind in "iu" and np.dtype(dtype).kind in "iu":
            a = a.view(dtype)
        else:
            a = a.astype(dtype)
    return np.ascontiguousarray(a)


def e4m3fn_to_double(code: int) -> float:
    """Value of one OCP E4M3FN byte (NaN for 0x7F/0xFF)."""
    return load().oracle_e4m3fn_to_double(code)


def decode(q, kv_cache, kv_scale, block_table, seq_lens, sm_scale, *, pos_mask=None,
           row_mask=None, threads: int = 0, lib=None, return_threads: bool = False):
    """Exact-definition MLA decode in FP64.

    For every request b, query position t and head h:
      n = seq_lens[b] - T + 1 + t visible positions (causal inside the draft);
      x_p = e4m3fn(code) * kv_scale, with position p read from page
      block_table[b][p // 64], row p % 64;
      s_p = sm_scale * sum_{d<576} q[b,t,h,d] * x_p[d];
      out = sum_p softmax(s)_p * x_p[:512];  lse = ln sum_p exp(s_p).
    ``pos_mask`` (length >= max seq_len) keeps only positions with mask 1, which
    yields the partial answer of that part of the history; ``row_mask``
    [B,T,H] computes only the selected rows (others stay 0 / NaN-free zeros).

    q: bf16 [B,T,H,576] (torch bf16 or int16 bit patterns); kv_cache: uint8
    [num_pages,64,576]; block_table int32 [B,max_pages]; seq_lens int32 [B].
    Returns (out float64 [B,T,H,512], lse float64 [B,T,H]).
    """
    lib = lib or load()
    qn = _np(q, np.int16)
    B, T, H, dq = qn.shape
    assert dq == D_QK
    kvn = _np(kv_cache, np.uint8)
    assert kvn.ndim == 3 and kvn.shape[1:] == (PAGE, D_QK)
    btn = _np(block_table, np.int32)
    sln = _np(seq_lens, np.int32)
    assert btn.shape[0] == B and sln.shape == (B,)
    out = np.zeros((B, T, H, D_V), dtype=np.float64)
    lse = np.zeros((B, T, H), dtype=np.float64)
    pm = _np(pos_mask, np.uint8) if pos_mask is not None else None
    rm = _np(row_mask, np.uint8) if row_mask is not None else None
    if rm is not None:
        assert rm.shape == (B, T, H)
    scale = float(_np(kv_scale, np.float32).reshape(-1)[0])
    rc = lib.oracle_mla_decode(
        qn.ctypes.data, kvn.ctypes.data, kvn.shape[0], scale, btn.ctypes.data,
        btn.shape[1], sln.ctypes.data, B, T, H, float(sm_scale),
        pm.ctypes.data if pm is not None else None, pm.shape[0] if pm is not None else 0,
        rm.ctypes.data if rm is not None else None, out.ctypes.data, lse.ctypes.data, threads)
    if rc < 0:
        raise ValueError(f"oracle_mla_decode failed with code {rc}")
    return (out, lse, rc) if return_threads else (out, lse)


def merge(part_out, part_lse, *, lib=None):
    """FP64 LSE merge of S partial answers: part_out [S,...,D], part_lse [S,...]."""
    lib = lib or load()
    po = _np(part_out, np.float64)
    pl = _np(part_lse, np.float64)
    S = po.shape[0]
    D = po.shape[-1]
    assert pl.shape == po.shape[:-1]
    rows = int(np.prod(pl.shape[1:])) if pl.ndim > 1 else 1
    out = np.zeros(po.shape[1:], dtype=np.float64)
    lse = np.zeros(pl.shape[1:], dtype=np.float64)
    rc = lib.oracle_lse_merge(S, rows, D, po.ctypes.data, pl.ctypes.data, out.ctypes.data,
                              lse.ctypes.data)
    if rc != 0:
        raise ValueError(f"oracle_lse_merge failed with code {rc}")
    return out, lse


def e4m3fn_encode(x, *, lib=None):
    """E4M3FN codes of binary32 values: clamp to +-448, round to nearest even,
    sign kept (NaN -> 0x7F).  Returns a uint8 array of x's shape."""
    lib = lib or load()
    xn = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    out = np.zeros(xn.shape, dtype=np.uint8)
    lib.oracle_e4m3fn_encode_array(xn.ctypes.data, xn.size, out.ctypes.data)
    return out


def append_latent(latent, kv_scale, block_table, start_pos, kv_cache, *, lib=None):
    """Append new latents to a copy of the paged cache and return it.

    latent: bf16 [B,T,576]; kv_scale: fp32 scalar; block_table int32 [B,max_pages];
    start_pos int32 [B] (position of latent[b,0] in request b's history);
    kv_cache uint8 [num_pages,64,576].  Position p = start_pos[b] + t gets the codes
    e4m3fn(latent[b,t,d] / kv_scale) (binary32 division) in page block_table[b][p//64],
    row p % 64.  Returns (new_cache uint8 array, status): status -2 if a row was
    skipped because its position or page id is out of range.
    """
    lib = lib or load()
    ln = _np(latent, np.int16)
    B, T, d = ln.shape
    assert d == D_QK
    btn = _np(block_table, np.int32)
    spn = _np(start_pos, np.int32)
    assert btn.shape[0] == B and spn.shape == (B,)
    kv = _np(kv_cache, np.uint8).copy()
    assert kv.ndim == 3 and kv.shape[1:] == (PAGE, D_QK)
    scale = float(_np(kv_scale, np.float32).reshape(-1)[0])
    rc = lib.oracle_append_latent(ln.ctypes.data, B, T, scale, btn.ctypes.data, btn.shape[1],
                                  btn.shape[1], spn.ctypes.data, kv.ctypes.data, kv.shape[0])
    if rc == -1:
        raise ValueError("oracle_append_latent: bad arguments")
    return kv, rc
