"""The allocation-free entry point, pl_nvfp4_lora_linear_static_ws (collected last).

It exists for callers that cannot allocate device memory (they get raw pointers
from a host program that owns every allocation, or must not call cudaMalloc on a
serving path), so it keeps its scratch in a library-owned device array instead of
a caller workspace.  Here it is called through the C ABI and must match the
workspace entry point, within the linear tolerance of the other tests, on two
calls in a row (the second call starts from whatever the first left in the shared
array); a problem too large for the array is refused before anything launches.  Both entry points
are also compared with the FP64 oracle on the oracle's own encoding of the weight.
"""

import ctypes

import numpy as np
import pytest
import torch

from precision_linear_gb300 import binding as pl
from precision_linear_gb300 import build
from oracle import linear as olin
from tests.gpu_cases import LINEAR_TOL, make_case, np32, oracle_quantize, to_dev_nvfp4

pytestmark = pytest.mark.gpu

_P = ctypes.c_void_p
_ARGTYPES = [_P, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, _P, _P, _P, _P, _P, ctypes.c_int,
             ctypes.c_float, _P, _P, ctypes.c_float, _P, ctypes.c_int, _P]


@pytest.fixture(scope="module")
def static_entry():
    build.build()
    fn = pl.lib().pl_nvfp4_lora_linear_static_ws
    fn.restype = ctypes.c_int
    fn.argtypes = _ARGTYPES
    return fn


def _ptr(t):
    return None if t is None else _P(t.data_ptr())


@pytest.mark.parametrize("d_o,d_i,M,r,norm", [
    (3584, 3584, 16, 32, True),   # tensor-core path, K split over a cluster
    (2048, 256, 64, 8, True),     # tensor-core path, one K chunk: no split
    (300, 272, 5, 8, False),      # generic CUDA-core path, no norm
])
def test_static_workspace_matches_workspace_entry(cuda_ok, static_entry, d_o, d_i, M, r, norm):
    case = make_case(d_o, d_i, M, r, seed=d_o + M)
    codes, scales, s_g = to_dev_nvfp4(*oracle_quantize(case["W"]))
    w_norm = case["w_norm"] if norm else None
    z = case["z"] if norm else None
    ref = pl.nvfp4_lora_linear(case["x"], codes, scales, s_g, case["A"], case["B"], 2.0, w_norm, z, 1e-6,
                               out_dtype=torch.float32)
    torch.cuda.synchronize()
    rms = float(torch.sqrt(torch.mean(ref.double() ** 2)))
    # the FP64 oracle on the same weights, for both entry points
    packed, sb, sg = oracle_quantize(case["W"])
    y_oracle = olin.nvfp4_lora_linear(np32(case["x"]).astype(np.float64), packed, sb, sg, np32(case["A"]),
                                      np32(case["B"]), 2.0, np32(w_norm) if norm else None,
                                      np32(z) if norm else None, 1e-6)
    rms_o = float(np.sqrt(np.mean(y_oracle ** 2)))
    stream = _P(torch.cuda.current_stream().cuda_stream)
    for call in range(2):
        y = torch.full((M, d_o), float("nan"), dtype=torch.float32, device="cuda")
        st = static_entry(_ptr(case["x"]), M, d_i, d_o, _ptr(codes), _ptr(scales), _ptr(s_g), _ptr(case["A"]),
                          _ptr(case["B"]), r, 2.0, _ptr(w_norm), _ptr(z), 1e-6, _ptr(y), pl.PL_DTYPE_F32, stream)
        assert st == 0, pl.status_string(st)
        torch.cuda.synchronize()
        err = float(torch.max(torch.abs(y.double() - ref.double())))
        assert np.isfinite(err) and err <= LINEAR_TOL * rms, (call, err, rms)
        err_o = float(np.max(np.abs(np32(y).astype(np.float64) - y_oracle)))
        assert err_o <= LINEAR_TOL * rms_o, (call, "vs oracle", err_o, rms_o)
    assert pl.last_device_status() == 0


def test_static_workspace_refuses_oversized_problem(cuda_ok, static_entry):
    # M = 64 at d_i = 65536 needs more scratch than the array holds: refused, nothing launched
    fake = _P(1 << 20)
    st = static_entry(fake, 64, 65536, 128, fake, fake, fake, None, None, 0, 0.0, None, None, 1e-6, fake,
                      pl.PL_DTYPE_BF16, None)
    assert st == 7  # PL_ERR_WORKSPACE
    assert pl.lib().pl_workspace_bytes(64, 65536, 128, 0) > (8 << 20)
