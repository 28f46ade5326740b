"""The Python binding's host-side checks, without a GPU: wrong dtypes, devices, ranks
and shapes are refused before anything reaches the library, and the AQN schedule
helpers map the library's sentinels to exceptions."""

import pytest
import torch

from precision_linear_gb300 import binding as pl


@pytest.fixture(scope="module", autouse=True)
def _built():
    from precision_linear_gb300 import build
    build.build()


def test_quantize_rejects_host_and_wrong_dtype():
    with pytest.raises(ValueError, match="CUDA"):
        pl.nvfp4_quantize(torch.zeros(16, 32, dtype=torch.bfloat16))
    with pytest.raises(TypeError, match="bfloat16"):
        pl.nvfp4_quantize(torch.zeros(16, 32, dtype=torch.float32))
    with pytest.raises(ValueError, match="CUDA"):
        pl.nvfp4_quantize_uaq(torch.zeros(16, 32, dtype=torch.bfloat16), 1.5)


def test_norm_and_linear_reject_host_tensors():
    x = torch.zeros(4, 256, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA"):
        pl.rmsnorm_aqn(x, torch.ones(256))
    with pytest.raises(ValueError, match="CUDA"):
        pl.uaq_fold_norm(torch.ones(256), 1.5)
    with pytest.raises((ValueError, TypeError)):
        pl.nvfp4_lora_linear(x, torch.zeros(256, 128, dtype=torch.uint8), torch.zeros(256, 16, dtype=torch.uint8),
                             torch.ones(1))


def test_noise_rejects_a_host_or_misshaped_output():
    with pytest.raises(ValueError, match="CUDA"):
        pl.aqn_noise(256, 1, out=torch.zeros(1, 256))
    with pytest.raises(TypeError):
        pl.aqn_noise(256, 1, out=torch.zeros(1, 256, dtype=torch.float64))


def test_schedule_helpers():
    assert pl.aqn_stage(0, 100) == 0 and pl.aqn_stage(100, 100) == 9
    assert pl.aqn_sigma(0, 0.01, 0.0005) == 0.0
    with pytest.raises(ValueError):
        pl.aqn_stage(1, 0)
    with pytest.raises(ValueError):
        pl.aqn_sigma(10, 0.01, 0.0005)
