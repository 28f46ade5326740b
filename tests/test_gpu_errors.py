"""Failure handling on the GPU without faulting it: an injected launch failure
is reported as PL_ERR_CUDA, and a bounded device wait that runs out is reported
as PL_ERR_TIMEOUT while the context stays usable."""

import pytest
import torch

from precision_linear_gb300 import binding as pl
from tests.gpu_cases import assert_linear_close, make_case, oracle_linear, oracle_quantize, to_dev_nvfp4

pytestmark = pytest.mark.gpu


def _linear(case, dev_w):
    return pl.nvfp4_lora_linear(case["x"], *dev_w, case["A"], case["B"], 2.0, case["w_norm"], case["z"],
                                out_dtype=torch.float32)


def test_injected_launch_failure_is_reported(cuda_ok):
    case = make_case(256, 256, 4, 8)
    dev_w = pl.nvfp4_quantize(case["W"])
    pl.lib().pl_debug_fail_next_launch(1)
    with pytest.raises(pl.PLError) as ei:
        _linear(case, dev_w)
    assert ei.value.status == 6
    _linear(case, dev_w)  # one-shot: the next call succeeds
    assert pl.last_device_status() == 0


def test_bounded_wait_timeout_is_reported_and_context_survives(cuda_ok):
    assert pl.last_device_status() == 0
    st = pl.lib().pl_debug_wait_timeout_probe(pl._stream(torch.device("cuda")))
    assert st == 0
    assert pl.last_device_status() == 8  # PL_ERR_TIMEOUT, read and cleared
    assert pl.last_device_status() == 0
    case = make_case(512, 512, 8, 8, seed=3)
    packed, sb, s_g = oracle_quantize(case["W"])
    y = _linear(case, to_dev_nvfp4(packed, sb, s_g))
    assert_linear_close(y, oracle_linear(case, packed, sb, s_g, 2.0), "after time-out probe")
