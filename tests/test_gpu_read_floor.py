"""fanout_read_floor, the calibration read that bench.py times beside an
HBM-bound call: it reads every byte of its buffer once (the xor of all the
buffer's words, checked against numpy on sizes that end inside the unrolled
step and one the size of the decode workload's K/V), through the C ABI."""
import numpy as np
import pytest
import torch

from shared_prefix_fan_gb300 import binding

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("nbytes", [16, 4096 + 48, (16 << 20) + 208, 151_060_480])
def test_read_floor_reads_every_word(nbytes):
    host = np.random.default_rng(nbytes).integers(0, 2**32, size=nbytes // 4, dtype=np.uint32)
    buf = torch.from_numpy(host.view(np.int32)).cuda()
    xo = torch.zeros(1, dtype=torch.int32, device="cuda")
    binding.read_floor(buf, xo)
    torch.cuda.synchronize()
    assert (int(xo.item()) & 0xFFFFFFFF) == int(np.bitwise_xor.reduce(host))
    binding.read_floor(buf, xo)   # twice: the xor cancels
    torch.cuda.synchronize()
    assert int(xo.item()) == 0


def test_read_floor_rejects_without_launching():
    buf = torch.zeros(1024, dtype=torch.uint8, device="cuda")
    xo = torch.zeros(1, dtype=torch.int32, device="cuda")
    lib = binding.load()
    assert lib.fanout_read_floor(buf.data_ptr() + 8, 512, xo.data_ptr(), None) == binding.EINVAL
    assert lib.fanout_read_floor(buf.data_ptr(), 40, xo.data_ptr(), None) == binding.EINVAL
    torch.cuda.synchronize()
    assert int(xo.item()) == 0
