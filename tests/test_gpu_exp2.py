"""The attention kernel's software exp2 (range reduction + fitted degree-3
polynomial) against CUDA's exp2 on the device: relative error within the
fit's bound over the whole input range the softmax produces."""
import pytest
import torch

from shared_prefix_fan_gb300 import binding, build

pytestmark = pytest.mark.gpu


def test_software_exp2_matches_cuda_exp2():
    build.build()
    x = torch.cat([torch.linspace(-126.0, 8.0, 2_000_001, device="cuda"),
                   torch.tensor([0.0, -0.5, 0.5, 7.999, -125.99], device="cuda")])
    y = binding.selftest_exp2(x)
    ref = torch.exp2(x.double())
    rel = (y.double() / ref - 1.0).abs()
    assert rel.max().item() <= 1.0e-4, rel.max().item()
    # exact powers of two stay within one polynomial error of exact
    xi = torch.arange(-120, 9, dtype=torch.float32, device="cuda")
    yi = binding.selftest_exp2(xi)
    assert ((yi.double() / torch.exp2(xi.double()) - 1).abs() <= 1e-4).all()
