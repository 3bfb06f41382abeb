"""The torch.optim front end rejects parameters the library cannot step
before it creates a device handle (no GPU needed)."""
import pytest
import torch

from muon_newton_schulz_gb300.optim import Muon


@pytest.mark.parametrize("shape, dtype, why", [
    ((8,), torch.float32, "2-D"),
    ((2, 3, 4), torch.float32, "2-D"),
    ((8, 8), torch.float16, "bf16 or fp32"),
    ((8, 8), torch.float32, "CUDA"),
])
def test_rejects_unsupported_parameters(shape, dtype, why):
    p = torch.nn.Parameter(torch.zeros(shape, dtype=dtype))
    with pytest.raises(ValueError, match=why):
        Muon([p])


def test_rejects_negative_lr():
    with pytest.raises(ValueError, match="learning rate"):
        Muon([torch.nn.Parameter(torch.zeros(4, 4))], lr=-1.0)
