"""spc_copy: the kernel copy the end-to-end loop uses for its host I/O, between
device memory and the device-visible address of pinned host memory, through
the C ABI. Bytes must arrive unchanged in every direction, aligned or not."""
import numpy as np
import pytest
import torch

from sparse_kv_cache_retrieval_gb300 import binding as spc

pytestmark = pytest.mark.gpu


def _bytes(n, seed):
    return torch.from_numpy(np.random.default_rng(seed).integers(0, 256, n, dtype=np.uint8))


@pytest.mark.parametrize("n", [0, 1, 15, 16, 4096 + 7, 3 << 20])
def test_host_to_device_and_back(n):
    src = _bytes(n, n).pin_memory()
    dev = torch.zeros(max(n, 1), dtype=torch.uint8, device="cuda")
    back = torch.zeros(max(n, 1), dtype=torch.uint8).pin_memory()
    if n:
        spc.spc_copy(dev, spc.spc_host_device_pointer(src), n)
        spc.spc_copy(spc.spc_host_device_pointer(back), dev, n)
    torch.cuda.synchronize()
    assert torch.equal(dev[:n].cpu(), src[:n])
    assert torch.equal(back[:n], src[:n])


@pytest.mark.parametrize("off_dst,off_src", [(0, 0), (1, 0), (0, 3), (5, 5), (16, 32)])
def test_device_to_device_any_alignment(off_dst, off_src):
    n = 100_003
    src = _bytes(n + 64, 7).cuda()
    dst = torch.zeros(n + 64, dtype=torch.uint8, device="cuda")
    spc.spc_copy(dst.data_ptr() + off_dst, src.data_ptr() + off_src, n)
    torch.cuda.synchronize()
    assert torch.equal(dst[off_dst:off_dst + n], src[off_src:off_src + n])
    assert int(dst[:off_dst].sum()) == 0 and int(dst[off_dst + n:].sum()) == 0


def test_rejects_null_pointers():
    with pytest.raises(spc.SpcError):
        spc.spc_copy(0, 0, 16)
