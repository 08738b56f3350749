"""The page-streaming probe behind bench.py's stream_ceiling: it runs, reads only
the pages it is given, and flags out-of-range page ids on the device."""
import pytest
import torch

pytestmark = pytest.mark.gpu

PAGE_ERR = 2  # device error code of a page id out of range


@pytest.fixture(scope="module")
def L():
    from mla_latent_kv_fp8_gb300 import build
    build.build()
    from mla_latent_kv_fp8_gb300 import _lib
    _lib.lib()
    return _lib


def test_stream_probe_runs_clean(L):
    kv = torch.randint(0, 255, (96, 64, 576), dtype=torch.uint8, device="cuda")
    g = torch.Generator().manual_seed(3)
    ids = torch.randperm(96, generator=g).to(torch.int32).cuda()
    assert L.mla_device_error() == 0
    for ctas, ppc in [(4, 24), (1, 96), (96, 1), (7, 13)]:
        L.mla_bench_stream_pages(kv, ids, ctas, ppc)
    torch.cuda.synchronize()
    assert L.mla_device_error() == 0


def test_stream_probe_flags_page_out_of_range(L):
    kv = torch.zeros((8, 64, 576), dtype=torch.uint8, device="cuda")
    ids = torch.tensor([0, 1, 8, 2], dtype=torch.int32, device="cuda")  # 8 is past the end
    L.mla_bench_stream_pages(kv, ids, 1, 4)
    torch.cuda.synchronize()
    assert L.mla_device_error() == PAGE_ERR
    assert L.mla_device_error() == 0
