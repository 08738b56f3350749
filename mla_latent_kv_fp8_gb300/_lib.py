"""ctypes binding of the C ABI in include/mla_decode.h (argument marshalling only).

Every function here has the same name and argument order as the C entry point
it wraps.  Tensors are torch tensors on the GPU; they are described to the
library by pointer, shape and strides, and the library launches its own CUDA
kernels on the given stream.  There is no fallback: if the compiled library
is missing, importing this module fails with an error that says how to build it.
"""
from __future__ import annotations

import ctypes
import os
import struct

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmla_decode.so")

MLA_OK = 0
STATUS = {0: "MLA_OK", 1: "MLA_ERR_INVALID_ARG", 2: "MLA_ERR_UNSUPPORTED", 3: "MLA_ERR_CUDA",
          4: "MLA_ERR_NO_MEMORY", 5: "MLA_ERR_DEVICE"}
IMPL_AUTO, IMPL_SIMT, IMPL_TCGEN05 = 0, 1, 2

_DTYPES = {torch.bfloat16: 1, torch.float32: 2, torch.uint8: 3, torch.float8_e4m3fn: 3, torch.int32: 4}

# Every symbol include/mla_decode.h declares.
EXPORTS = ("mla_decode_paged", "mla_merge_partials", "mla_auto_splits", "mla_split_chunk_pages",
           "mla_decode_workspace_bytes", "mla_set_impl", "mla_device_error", "mla_status_string",
           "mla_last_error", "mla_profile_next_decode", "mla_last_decode_impl",
           "mla_decode_paged_noalloc", "mla_test_stall_copies", "mla_bench_stream_pages",
           "mla_append_latent", "mla_plan_splits", "mla_test_count_rescales",
           "mla_release_graph_scratch")


class MlaError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS.get(status, status)}: {message}")
        self.status = status


class mla_tensor_t(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("shape", ctypes.c_int64 * 5),
                ("stride", ctypes.c_int64 * 5), ("ndim", ctypes.c_int32), ("dtype", ctypes.c_int32)]


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    if not os.path.exists(path):
        raise ImportError(f"{path} is missing: build it with `python -c \"import __graft_entry__ as g; "
                          f"g.build()\"` (nvcc, sm_103a)")
    lib = ctypes.CDLL(path)
    if ctypes.sizeof(mla_tensor_t) != _DESC.size:
        raise ImportError("mla_tensor_t layout does not match the packed descriptor")
    P, T = ctypes.c_void_p, ctypes.POINTER(mla_tensor_t)
    lib.mla_decode_paged.argtypes = [T, T, P, T, T, ctypes.c_int32, ctypes.c_float, T, T, P]
    lib.mla_decode_paged.restype = ctypes.c_int
    lib.mla_decode_paged_noalloc.argtypes = [T, T, P, T, T, ctypes.c_int32, ctypes.c_float, T, T, P]
    lib.mla_decode_paged_noalloc.restype = ctypes.c_int
    lib.mla_append_latent.argtypes = [T, P, T, T, T, P]
    lib.mla_append_latent.restype = ctypes.c_int
    lib.mla_merge_partials.argtypes = [T, T, ctypes.c_int32, T, T, P]
    lib.mla_merge_partials.restype = ctypes.c_int
    lib.mla_auto_splits.argtypes = [ctypes.c_int32] * 5
    lib.mla_auto_splits.restype = ctypes.c_int32
    lib.mla_plan_splits.argtypes = [ctypes.c_int32] * 3 + [ctypes.POINTER(ctypes.c_int32)] + [ctypes.c_int32] * 2
    lib.mla_plan_splits.restype = ctypes.c_int32
    lib.mla_split_chunk_pages.argtypes = [ctypes.c_int32, ctypes.c_int32]
    lib.mla_split_chunk_pages.restype = ctypes.c_int32
    lib.mla_decode_workspace_bytes.argtypes = [ctypes.c_int32] * 4
    lib.mla_decode_workspace_bytes.restype = ctypes.c_size_t
    lib.mla_set_impl.argtypes = [ctypes.c_int32]
    lib.mla_set_impl.restype = ctypes.c_int32
    lib.mla_test_stall_copies.argtypes = [ctypes.c_int]
    lib.mla_test_stall_copies.restype = ctypes.c_int
    lib.mla_test_count_rescales.argtypes = [P]
    lib.mla_test_count_rescales.restype = ctypes.c_int
    lib.mla_release_graph_scratch.argtypes = []
    lib.mla_release_graph_scratch.restype = ctypes.c_int
    lib.mla_bench_stream_pages.argtypes = [P, ctypes.c_int64, P, ctypes.c_int32, ctypes.c_int32, P]
    lib.mla_bench_stream_pages.restype = ctypes.c_int
    lib.mla_device_error.argtypes = [ctypes.POINTER(ctypes.c_int32), P]
    lib.mla_device_error.restype = ctypes.c_int
    lib.mla_last_decode_impl.argtypes = []
    lib.mla_last_decode_impl.restype = ctypes.c_int32
    lib.mla_profile_next_decode.argtypes = [P, P]
    lib.mla_profile_next_decode.restype = ctypes.c_int
    lib.mla_status_string.argtypes = [ctypes.c_int]
    lib.mla_status_string.restype = ctypes.c_char_p
    lib.mla_last_error.argtypes = []
    lib.mla_last_error.restype = ctypes.c_char_p
    return lib


_lib = None


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        _lib = load_library()
    return _lib


_DESC = struct.Struct("<Q5q5qii")  # the byte layout of mla_tensor_t
_PAD = tuple((0,) * k for k in range(6))


def describe(t: torch.Tensor | None):
    """torch tensor -> mla_tensor_t (no copy; the tensor must outlive the call)."""
    if t is None:
        return None
    n = t.dim()
    if n > 5:
        raise ValueError("at most 5 dims")
    pad = _PAD[5 - n]
    return mla_tensor_t.from_buffer_copy(_DESC.pack(t.data_ptr(), *t.shape, *pad, *t.stride(), *pad, n,
                                                    _DTYPES.get(t.dtype, 0)))


def _ref(d):
    return ctypes.byref(d) if d is not None else None


def _stream(stream):
    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _check(status: int):
    if status != MLA_OK:
        raise MlaError(status, lib().mla_last_error().decode())


def mla_decode_paged(q, kv_cache, kv_scale, block_table, seq_lens, n_splits, sm_scale, out,
                     lse=None, stream=None):
    """out[b,t,h] = softmax(q . x^T * sm_scale) . x[:, :512] over the paged FP8 history."""
    dq, dkv, dbt, dsl, do, dl = (describe(q), describe(kv_cache), describe(block_table),
                                 describe(seq_lens), describe(out), describe(lse))
    _check(lib().mla_decode_paged(_ref(dq), _ref(dkv), ctypes.c_void_p(kv_scale.data_ptr()),
                                  _ref(dbt), _ref(dsl), int(n_splits), float(sm_scale), _ref(do),
                                  _ref(dl), _stream(stream)))


def mla_decode_paged_noalloc(q, kv_cache, kv_scale, block_table, seq_lens, n_splits, sm_scale, out,
                             lse=None, stream=None):
    """mla_decode_paged with its split scratch in the library's fixed 8 MiB device array."""
    dq, dkv, dbt, dsl, do, dl = (describe(q), describe(kv_cache), describe(block_table),
                                 describe(seq_lens), describe(out), describe(lse))
    _check(lib().mla_decode_paged_noalloc(_ref(dq), _ref(dkv), ctypes.c_void_p(kv_scale.data_ptr()),
                                          _ref(dbt), _ref(dsl), int(n_splits), float(sm_scale),
                                          _ref(do), _ref(dl), _stream(stream)))


def mla_append_latent(latent, kv_scale, block_table, start_pos, kv_cache, stream=None):
    """Quantise latent [B, T, 576] (bf16) to e4m3fn(x / kv_scale) and write position
    start_pos[b] + t of each request into its paged slot of kv_cache, in place."""
    dl, dbt, dsp, dkv = describe(latent), describe(block_table), describe(start_pos), describe(kv_cache)
    _check(lib().mla_append_latent(_ref(dl), ctypes.c_void_p(kv_scale.data_ptr()), _ref(dbt), _ref(dsp),
                                   _ref(dkv), _stream(stream)))


def mla_merge_partials(partial_out, partial_lse, n_shards, out, lse=None, stream=None):
    """Merge S partial answers [S, ..., 512] by their log-sum-exp normalisers."""
    dpo, dpl, do, dl = describe(partial_out), describe(partial_lse), describe(out), describe(lse)
    _check(lib().mla_merge_partials(_ref(dpo), _ref(dpl), int(n_shards), _ref(do), _ref(dl),
                                    _stream(stream)))


def mla_auto_splits(B, T, H, max_pages, sm_count=0):
    return lib().mla_auto_splits(B, T, H, max_pages, sm_count)


def mla_plan_splits(B, T, H, host_seq_lens, max_pages, sm_count=0):
    """host_seq_lens: B lengths on the host (a sequence of ints, or a CPU int32
    tensor / array)."""
    arr = (ctypes.c_int32 * B)(*[int(x) for x in host_seq_lens])
    return lib().mla_plan_splits(B, T, H, arr, max_pages, sm_count)


def mla_split_chunk_pages(max_pages, n_splits):
    return lib().mla_split_chunk_pages(max_pages, n_splits)


def mla_decode_workspace_bytes(B, T, H, n_splits):
    return lib().mla_decode_workspace_bytes(B, T, H, n_splits)


def mla_set_impl(impl: int) -> int:
    return lib().mla_set_impl(impl)


def mla_test_stall_copies(on: bool) -> int:
    """Failure-detection tests only: later tensor-core launches from this thread
    issue no page copies, so their bounded waits run out (device error 1).
    Returns the previous setting of this thread."""
    return lib().mla_test_stall_copies(1 if on else 0)


def mla_test_count_rescales(device_counts):
    """The next decode call of this thread adds to device_counts (a zeroed int32
    CUDA tensor of 2): [0] in-place rescales of accumulated output tiles after a
    warpgroup's first page, [1] reference moves of any kind."""
    _check(lib().mla_test_count_rescales(ctypes.c_void_p(device_counts.data_ptr())))


def mla_release_graph_scratch():
    """Free the split scratch kept for captured CUDA graphs on the current device
    (only once no such graph will be replayed)."""
    _check(lib().mla_release_graph_scratch())


def mla_bench_stream_pages(kv_cache, page_ids, ctas, pages_per_cta, stream=None):
    """Benchmark instrumentation: stream the given pages of the cache through the
    decode kernel's TMA ring with no arithmetic (the HBM ceiling of that pattern)."""
    _check(lib().mla_bench_stream_pages(ctypes.c_void_p(kv_cache.data_ptr()), int(kv_cache.shape[0]),
                                        ctypes.c_void_p(page_ids.data_ptr()), int(ctas), int(pages_per_cta),
                                        _stream(stream)))


def mla_last_decode_impl() -> int:
    return lib().mla_last_decode_impl()


def mla_device_error(stream=None) -> int:
    code = ctypes.c_int32(0)
    _check(lib().mla_device_error(ctypes.byref(code), _stream(stream)))
    return code.value


def mla_profile_next_decode(ev_begin, ev_end):
    """Record raw cudaEvent_t handles (ints) around the next decode kernel of this thread."""
    _check(lib().mla_profile_next_decode(ctypes.c_void_p(ev_begin or 0), ctypes.c_void_p(ev_end or 0)))


def mla_status_string(status: int) -> str:
    return lib().mla_status_string(status).decode()


def mla_last_error() -> str:
    return lib().mla_last_error().decode()
