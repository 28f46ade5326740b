"""ctypes binding of libprecision_linear.so: argument marshalling only.

Every step of the path runs in the library's CUDA kernels; this module checks
tensor dtypes/devices, allocates outputs with torch when the caller does not pass
them, hands raw device pointers and the current torch stream to the C ABI, and
turns non-zero status codes into ``PLError``.  There is no fallback: if the
library is missing or the device is not sm_103, calls raise.
"""

from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libprecision_linear.so")

_c_void_p = ctypes.c_void_p
_i64 = ctypes.c_int64
_lock = threading.Lock()
_lib = None

PL_OK = 0
PL_DTYPE_BF16 = 0
PL_DTYPE_F32 = 1
_OUT_DTYPES = {torch.bfloat16: PL_DTYPE_BF16, torch.float32: PL_DTYPE_F32}


class PLError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = int(status)
        super().__init__(f"{where}: {status_string(status)}")


class Proj(ctypes.Structure):
    """pl_nvfp4_proj: one projection of a group call."""
    _fields_ = [("d_o", ctypes.c_int64), ("codes", ctypes.c_void_p), ("scales", ctypes.c_void_p),
                ("s_g", ctypes.c_void_p), ("A", ctypes.c_void_p), ("B", ctypes.c_void_p), ("r", ctypes.c_int),
                ("lam", ctypes.c_float), ("y", ctypes.c_void_p)]


class Call(ctypes.Structure):
    """pl_nvfp4_call: one call of a batch."""
    _fields_ = [("x", ctypes.c_void_p), ("M", ctypes.c_int64), ("d_o", ctypes.c_int64), ("codes", ctypes.c_void_p),
                ("scales", ctypes.c_void_p), ("s_g", ctypes.c_void_p), ("A", ctypes.c_void_p), ("B", ctypes.c_void_p),
                ("r", ctypes.c_int), ("lam", ctypes.c_float), ("w_norm", ctypes.c_void_p), ("z", ctypes.c_void_p),
                ("z_ld", ctypes.c_int64), ("y", ctypes.c_void_p)]


_SIGNATURES = {
    "pl_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "pl_version": (ctypes.c_int, []),
    "pl_nvfp4_bytes": (ctypes.c_size_t, [_i64, _i64]),
    "pl_workspace_bytes": (ctypes.c_size_t, [_i64, _i64, _i64, ctypes.c_int]),
    "pl_nvfp4_quantize": (ctypes.c_int, [_c_void_p, _i64, _i64, _c_void_p, _c_void_p, _c_void_p, _c_void_p]),
    "pl_rmsnorm_aqn": (ctypes.c_int, [_c_void_p, _i64, _i64, _c_void_p, _c_void_p, _i64, ctypes.c_float,
                                      _c_void_p, ctypes.c_int, _c_void_p]),
    "pl_nvfp4_lora_linear": (ctypes.c_int, [_c_void_p, _i64, _i64, _i64, _c_void_p, _c_void_p, _c_void_p,
                                            _c_void_p, _c_void_p, ctypes.c_int, ctypes.c_float,
                                            _c_void_p, _c_void_p, _i64, ctypes.c_float, _c_void_p, ctypes.c_int,
                                            _c_void_p, ctypes.c_size_t, _c_void_p]),
    "pl_workspace_bytes_group": (ctypes.c_size_t, [_i64, _i64, ctypes.POINTER(Proj), ctypes.c_int]),
    "pl_nvfp4_lora_linear_group": (ctypes.c_int, [_c_void_p, _i64, _i64, _c_void_p, _c_void_p, _i64, ctypes.c_float,
                                                  ctypes.POINTER(Proj), ctypes.c_int, ctypes.c_int, _c_void_p,
                                                  ctypes.c_size_t, _c_void_p]),
    "pl_workspace_bytes_batch": (ctypes.c_size_t, [_i64, ctypes.POINTER(Call), ctypes.c_int]),
    "pl_nvfp4_lora_linear_batch": (ctypes.c_int, [_i64, ctypes.c_float, ctypes.POINTER(Call), ctypes.c_int,
                                                  ctypes.c_int, _c_void_p, ctypes.c_size_t, _c_void_p]),
    "pl_w8a8_workspace_bytes": (ctypes.c_size_t, [_i64, _i64, _i64, ctypes.c_int]),
    "pl_w8a8_quantize_weight": (ctypes.c_int, [_c_void_p, _i64, _i64, _c_void_p, _c_void_p, _c_void_p]),
    "pl_w8a8_lora_linear": (ctypes.c_int, [_c_void_p, _i64, _i64, _i64, _c_void_p, _c_void_p, _c_void_p, _c_void_p,
                                           ctypes.c_int, ctypes.c_float, _c_void_p, _c_void_p, _i64, ctypes.c_float,
                                           _c_void_p, ctypes.c_int, _c_void_p, ctypes.c_size_t, _c_void_p]),
    "pl_backward_workspace_bytes": (ctypes.c_size_t, [_i64, _i64, _i64, ctypes.c_int, ctypes.c_int]),
    "pl_nvfp4_lora_linear_backward": (ctypes.c_int, [_c_void_p, _i64, _i64, _i64, _c_void_p, _c_void_p, _c_void_p,
                                                     _c_void_p, _c_void_p, ctypes.c_int, ctypes.c_float, _c_void_p,
                                                     _c_void_p, _c_void_p, _i64, ctypes.c_float, _c_void_p,
                                                     _c_void_p, _c_void_p, _c_void_p, ctypes.c_size_t, _c_void_p]),
    "pl_nvfp4_quantize_uaq": (ctypes.c_int, [_c_void_p, _i64, _i64, ctypes.c_float, _c_void_p, _c_void_p,
                                             _c_void_p, _c_void_p]),
    "pl_uaq_fold_norm": (ctypes.c_int, [_c_void_p, _i64, ctypes.c_float, _c_void_p, _c_void_p]),
    "pl_aqn_stage": (ctypes.c_int, [_i64, _i64]),
    "pl_aqn_sigma": (ctypes.c_float, [ctypes.c_int, ctypes.c_float, ctypes.c_float]),
    "pl_aqn_noise": (ctypes.c_int, [ctypes.c_uint64, ctypes.c_uint32, ctypes.c_uint64, _i64, _i64, ctypes.c_float,
                                    _c_void_p, _c_void_p]),
    "pl_last_device_status": (ctypes.c_int, [_c_void_p]),
    "pl_debug_fail_next_launch": (None, [ctypes.c_int]),
    "pl_debug_linear_path": (ctypes.c_int, [_i64, _i64, _i64, ctypes.c_int]),
    "pl_debug_wait_timeout_probe": (ctypes.c_int, [_c_void_p]),
}


def lib() -> ctypes.CDLL:
    """The loaded shared library (loaded once)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"{LIB_PATH} is not built: run `python -m precision_linear_gb300.build`")
            L = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in _SIGNATURES.items():
                fn = getattr(L, name)
                fn.restype = res
                fn.argtypes = args
            _lib = L
    return _lib


def status_string(status: int) -> str:
    try:
        return lib().pl_status_string(int(status)).decode()
    except Exception:  # library not loadable
        return f"status {status}"


def _check(status: int, where: str):
    if status != PL_OK:
        raise PLError(status, where)


def _ptr(t):
    return None if t is None else _c_void_p(t.data_ptr())


def _stream(device) -> _c_void_p:
    return _c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _need(t, name, dtype, device=None, dim=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if dim is not None and t.dim() != dim:
        raise ValueError(f"{name} must be {dim}-D")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _noise(z, M: int, d: int, dev):
    """(z, z_ld) for the C ABI: a [d] vector is every row's state (z_ld = 0); a [M, d]
    tensor (row stride a multiple of 4, unit column stride) gives row m its own state."""
    if z is None:
        return None, 0
    if not isinstance(z, torch.Tensor) or z.dtype != torch.float32 or not z.is_cuda or z.device != dev:
        raise TypeError(f"z must be a float32 tensor on {dev}")
    if z.dim() == 1:
        if z.shape[0] != d or not z.is_contiguous():
            raise ValueError(f"z must be a contiguous vector of {d} elements")
        return z, 0
    if z.dim() != 2 or tuple(z.shape) != (M, d) or z.stride(1) != 1 or z.stride(0) < d or z.stride(0) % 4:
        raise ValueError(f"per-row z must be [{M}, {d}] with unit column stride and a row stride that is a "
                         "multiple of 4")
    return z, int(z.stride(0))


def nvfp4_bytes(d_o: int, d_i: int) -> int:
    return int(lib().pl_nvfp4_bytes(d_o, d_i))


def workspace_bytes(M: int, d_i: int, d_o: int, r: int) -> int:
    return int(lib().pl_workspace_bytes(M, d_i, d_o, r))


def nvfp4_quantize(W: torch.Tensor, codes=None, scales=None, s_g=None):
    """BF16 W [d_o, d_i] -> (codes uint8 [d_o, d_i/2], scales uint8 [d_o, d_i/16], s_g float32 [1])."""
    _need(W, "W", torch.bfloat16, dim=2)
    d_o, d_i = W.shape
    dev = W.device
    if codes is None:
        codes = torch.empty(d_o, d_i // 2, dtype=torch.uint8, device=dev)
    if scales is None:
        scales = torch.empty(d_o, max(d_i // 16, 1), dtype=torch.uint8, device=dev)
    if s_g is None:
        s_g = torch.empty(1, dtype=torch.float32, device=dev)
    with torch.cuda.device(dev):
        st = lib().pl_nvfp4_quantize(_ptr(W), d_o, d_i, _ptr(codes), _ptr(scales), _ptr(s_g), _stream(dev))
    _check(st, "pl_nvfp4_quantize")
    return codes, scales, s_g


def nvfp4_quantize_uaq(W: torch.Tensor, s: float = 1.5, codes=None, scales=None, s_g=None):
    """NVFP4 encoding of fp32(W / s) (the UAQ fold's weight half); returns (codes, scales, s_g)."""
    _need(W, "W", torch.bfloat16, dim=2)
    d_o, d_i = W.shape
    dev = W.device
    if codes is None:
        codes = torch.empty(d_o, d_i // 2, dtype=torch.uint8, device=dev)
    if scales is None:
        scales = torch.empty(d_o, max(d_i // 16, 1), dtype=torch.uint8, device=dev)
    if s_g is None:
        s_g = torch.empty(1, dtype=torch.float32, device=dev)
    with torch.cuda.device(dev):
        st = lib().pl_nvfp4_quantize_uaq(_ptr(W), d_o, d_i, float(s), _ptr(codes), _ptr(scales), _ptr(s_g),
                                         _stream(dev))
    _check(st, "pl_nvfp4_quantize_uaq")
    return codes, scales, s_g


def uaq_fold_norm(w_norm: torch.Tensor, s: float = 1.5, out: torch.Tensor | None = None) -> torch.Tensor:
    """fp32(w_norm * s) (the UAQ fold's norm half)."""
    _need(w_norm, "w_norm", torch.float32, dim=1)
    dev = w_norm.device
    if out is None:
        out = torch.empty_like(w_norm)
    _need(out, "out", torch.float32, dev, 1)
    with torch.cuda.device(dev):
        st = lib().pl_uaq_fold_norm(_ptr(w_norm), w_norm.numel(), float(s), _ptr(out), _stream(dev))
    _check(st, "pl_uaq_fold_norm")
    return out


def rmsnorm_aqn(x: torch.Tensor, w_norm: torch.Tensor, z: torch.Tensor | None = None,
                eps: float = 1e-6, out: torch.Tensor | None = None,
                out_dtype: torch.dtype = torch.bfloat16) -> torch.Tensor:
    """h = x / sqrt(mean(x^2) + eps) * (w_norm + z_m) per row m, BF16 or FP32 output.
    z: None, one [d] vector for every row, or [M, d] (one noise state per row)."""
    _need(x, "x", torch.bfloat16, dim=2)
    dev = x.device
    _need(w_norm, "w_norm", torch.float32, dev, 1)
    z, z_ld = _noise(z, x.shape[0], x.shape[1], dev)
    if out is None:
        out = torch.empty(x.shape, dtype=out_dtype, device=dev)
    _need(out, "out", out.dtype, dev, 2)
    if out.dtype not in _OUT_DTYPES:
        raise TypeError("out must be bfloat16 or float32")
    M, d = x.shape
    with torch.cuda.device(dev):
        st = lib().pl_rmsnorm_aqn(_ptr(x), M, d, _ptr(w_norm), _ptr(z), z_ld, float(eps), _ptr(out),
                                  _OUT_DTYPES[out.dtype], _stream(dev))
    _check(st, "pl_rmsnorm_aqn")
    return out


class Workspace:
    """A growable device scratch buffer for pl_nvfp4_lora_linear (one per stream)."""

    def __init__(self, device=None):
        self.device = torch.device(device) if device is not None else torch.device("cuda")
        self.buf = None

    def get(self, nbytes: int) -> torch.Tensor:
        if self.buf is None or self.buf.numel() < nbytes:
            self.buf = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=self.device)
        return self.buf


_default_ws = {}


def nvfp4_lora_linear(x, codes, scales, s_g, A=None, B=None, lam: float = 0.0, w_norm=None, z=None,
                      eps: float = 1e-6, out=None, workspace: Workspace | None = None,
                      out_dtype: torch.dtype = torch.bfloat16) -> torch.Tensor:
    """y = W_hat h + lam * B (A h) with h = RMSNorm_AQN(x) when w_norm is given (else x).
    z: None, one [d_i] noise vector for every row, or [M, d_i] (one noise state per row)."""
    _need(x, "x", torch.bfloat16, dim=2)
    dev = x.device
    _need(codes, "codes", torch.uint8, dev, 2)
    _need(scales, "scales", torch.uint8, dev, 2)
    _need(s_g, "s_g", torch.float32, dev)
    M, d_i = x.shape
    d_o = codes.shape[0]
    r = 0
    if A is not None or B is not None:
        _need(A, "A", torch.bfloat16, dev, 2)
        _need(B, "B", torch.bfloat16, dev, 2)
        r = A.shape[0]
    if w_norm is not None:
        _need(w_norm, "w_norm", torch.float32, dev, 1)
    z, z_ld = _noise(z, M, d_i, dev)
    if out is None:
        out = torch.empty(M, d_o, dtype=out_dtype, device=dev)
    if out.dtype not in _OUT_DTYPES:
        raise TypeError("out must be bfloat16 or float32")
    _need(out, "out", out.dtype, dev, 2)
    need = workspace_bytes(M, d_i, d_o, r)
    if workspace is None:
        workspace = _default_ws.setdefault(dev, Workspace(dev))
    ws = workspace.get(need)
    with torch.cuda.device(dev):
        st = lib().pl_nvfp4_lora_linear(_ptr(x), M, d_i, d_o, _ptr(codes), _ptr(scales), _ptr(s_g),
                                        _ptr(A), _ptr(B), r, float(lam), _ptr(w_norm), _ptr(z), z_ld, float(eps),
                                        _ptr(out), _OUT_DTYPES[out.dtype], _ptr(ws), ws.numel(), _stream(dev))
    _check(st, "pl_nvfp4_lora_linear")
    return out


def nvfp4_lora_linear_group(x, projs, w_norm=None, z=None, eps: float = 1e-6, outs=None,
                            workspace: Workspace | None = None, out_dtype: torch.dtype = torch.bfloat16):
    """The projections that read one input (e.g. q/k/v behind one RMSNorm) in one call.

    projs: sequence of dicts with keys codes, scales, s_g and optionally A, B, lam; every
    projection gets y_p = W_hat_p h + lam_p B_p (A_p h) with the shared h = RMSNorm_AQN(x)
    (x when w_norm is None).  Returns the list of y_p."""
    _need(x, "x", torch.bfloat16, dim=2)
    dev = x.device
    M, d_i = x.shape
    if w_norm is not None:
        _need(w_norm, "w_norm", torch.float32, dev, 1)
    z, z_ld = _noise(z, M, d_i, dev)
    n = len(projs)
    arr = (Proj * max(n, 1))()
    ys = []
    for i, q in enumerate(projs):
        codes, scales, s_g = q["codes"], q["scales"], q["s_g"]
        _need(codes, "codes", torch.uint8, dev, 2)
        _need(scales, "scales", torch.uint8, dev, 2)
        _need(s_g, "s_g", torch.float32, dev)
        A, B = q.get("A"), q.get("B")
        r = 0
        if A is not None or B is not None:
            _need(A, "A", torch.bfloat16, dev, 2)
            _need(B, "B", torch.bfloat16, dev, 2)
            r = A.shape[0]
        d_o = codes.shape[0]
        y = outs[i] if outs is not None else torch.empty(M, d_o, dtype=out_dtype, device=dev)
        if y.dtype != out_dtype:
            raise TypeError("every output of a group has the group's dtype")
        _need(y, "out", out_dtype, dev, 2)
        ys.append(y)
        arr[i] = Proj(d_o, codes.data_ptr(), scales.data_ptr(), s_g.data_ptr(), A.data_ptr() if A is not None else None,
                      B.data_ptr() if B is not None else None, r, float(q.get("lam", 0.0)), y.data_ptr())
    if out_dtype not in _OUT_DTYPES:
        raise TypeError("out_dtype must be bfloat16 or float32")
    need = int(lib().pl_workspace_bytes_group(M, d_i, arr, n))
    if workspace is None:
        workspace = _default_ws.setdefault(dev, Workspace(dev))
    ws = workspace.get(max(need, 256))
    with torch.cuda.device(dev):
        st = lib().pl_nvfp4_lora_linear_group(_ptr(x), M, d_i, _ptr(w_norm), _ptr(z), z_ld, float(eps), arr, n,
                                              _OUT_DTYPES[out_dtype], _ptr(ws), ws.numel(), _stream(dev))
    _check(st, "pl_nvfp4_lora_linear_group")
    return ys


def nvfp4_lora_linear_batch(calls, eps: float = 1e-6, outs=None, workspace: Workspace | None = None,
                            out_dtype: torch.dtype = torch.bfloat16):
    """Independent calls of the linear in one batch: calls is a sequence of dicts with keys x,
    codes, scales, s_g and optionally A, B, lam, w_norm, z (as nvfp4_lora_linear's arguments);
    every call has the same d_i.  Returns the list of y."""
    n = len(calls)
    arr = (Call * max(n, 1))()
    ys, keep = [], []
    d_i = None
    for i, c in enumerate(calls):
        x = c["x"]
        _need(x, "x", torch.bfloat16, dim=2)
        dev = x.device
        M, di = x.shape
        if d_i is None:
            d_i = di
        elif di != d_i:
            raise ValueError("every call of a batch has the same d_i")
        codes, scales, s_g = c["codes"], c["scales"], c["s_g"]
        _need(codes, "codes", torch.uint8, dev, 2)
        _need(scales, "scales", torch.uint8, dev, 2)
        _need(s_g, "s_g", torch.float32, dev)
        A, B = c.get("A"), c.get("B")
        r = 0
        if A is not None or B is not None:
            _need(A, "A", torch.bfloat16, dev, 2)
            _need(B, "B", torch.bfloat16, dev, 2)
            r = A.shape[0]
        w = c.get("w_norm")
        if w is not None:
            _need(w, "w_norm", torch.float32, dev, 1)
        z, z_ld = _noise(c.get("z"), M, d_i, dev)
        d_o = codes.shape[0]
        y = outs[i] if outs is not None else torch.empty(M, d_o, dtype=out_dtype, device=dev)
        _need(y, "out", out_dtype, dev, 2)
        ys.append(y)
        keep.append(z)
        arr[i] = Call(x.data_ptr(), M, d_o, codes.data_ptr(), scales.data_ptr(), s_g.data_ptr(),
                      A.data_ptr() if A is not None else None, B.data_ptr() if B is not None else None, r,
                      float(c.get("lam", 0.0)), w.data_ptr() if w is not None else None,
                      z.data_ptr() if z is not None else None, z_ld, y.data_ptr())
    if out_dtype not in _OUT_DTYPES:
        raise TypeError("out_dtype must be bfloat16 or float32")
    dev = calls[0]["x"].device
    need = int(lib().pl_workspace_bytes_batch(d_i, arr, n))
    if workspace is None:
        workspace = _default_ws.setdefault(dev, Workspace(dev))
    ws = workspace.get(max(need, 256))
    with torch.cuda.device(dev):
        st = lib().pl_nvfp4_lora_linear_batch(d_i, float(eps), arr, n, _OUT_DTYPES[out_dtype], _ptr(ws), ws.numel(),
                                              _stream(dev))
    _check(st, "pl_nvfp4_lora_linear_batch")
    return ys


def w8a8_quantize_weight(W: torch.Tensor, codes=None, s_w=None):
    """BF16 W [d_o, d_i] -> (E4M3 codes uint8 [d_o, d_i], s_w float32 [d_o]): one FP8 scale per
    output channel (the W8A8 rollout linear's weight)."""
    _need(W, "W", torch.bfloat16, dim=2)
    d_o, d_i = W.shape
    dev = W.device
    if codes is None:
        codes = torch.empty(d_o, d_i, dtype=torch.uint8, device=dev)
    if s_w is None:
        s_w = torch.empty(d_o, dtype=torch.float32, device=dev)
    with torch.cuda.device(dev):
        st = lib().pl_w8a8_quantize_weight(_ptr(W), d_o, d_i, _ptr(codes), _ptr(s_w), _stream(dev))
    _check(st, "pl_w8a8_quantize_weight")
    return codes, s_w


def w8a8_lora_linear(x, codes, s_w, A=None, B=None, lam: float = 0.0, w_norm=None, z=None, eps: float = 1e-6,
                     out=None, workspace: Workspace | None = None, out_dtype: torch.dtype = torch.bfloat16):
    """y = s_x s_w (q_x q_w^T) + lam * B (A h), h = RMSNorm_AQN(x) (x when w_norm is None),
    q_x the per-token FP8 quantisation of h."""
    _need(x, "x", torch.bfloat16, dim=2)
    dev = x.device
    _need(codes, "codes", torch.uint8, dev, 2)
    _need(s_w, "s_w", torch.float32, dev, 1)
    M, d_i = x.shape
    d_o = codes.shape[0]
    r = 0
    if A is not None or B is not None:
        _need(A, "A", torch.bfloat16, dev, 2)
        _need(B, "B", torch.bfloat16, dev, 2)
        r = A.shape[0]
    if w_norm is not None:
        _need(w_norm, "w_norm", torch.float32, dev, 1)
    z, z_ld = _noise(z, M, d_i, dev)
    if out is None:
        out = torch.empty(M, d_o, dtype=out_dtype, device=dev)
    if out.dtype not in _OUT_DTYPES:
        raise TypeError("out must be bfloat16 or float32")
    _need(out, "out", out.dtype, dev, 2)
    need = int(lib().pl_w8a8_workspace_bytes(M, d_i, d_o, r))
    if workspace is None:
        workspace = _default_ws.setdefault(dev, Workspace(dev))
    ws = workspace.get(max(need, 256))
    with torch.cuda.device(dev):
        st = lib().pl_w8a8_lora_linear(_ptr(x), M, d_i, d_o, _ptr(codes), _ptr(s_w), _ptr(A), _ptr(B), r, float(lam),
                                       _ptr(w_norm), _ptr(z), z_ld, float(eps), _ptr(out), _OUT_DTYPES[out.dtype],
                                       _ptr(ws), ws.numel(), _stream(dev))
    _check(st, "pl_w8a8_lora_linear")
    return out


def nvfp4_lora_linear_backward(g, x, codes, scales, s_g, A=None, B=None, lam: float = 0.0, w_norm=None, z=None,
                               eps: float = 1e-6, want_adapter_grads: bool = True, workspace: Workspace | None = None):
    """Gradients of the frozen-backbone linear for dL/dy = g (BF16 [M, d_o]): returns
    (dx FP32 [M, d_i], dA FP32 [r, d_i] or None, dB FP32 [d_o, r] or None)."""
    _need(g, "g", torch.bfloat16, dim=2)
    dev = g.device
    _need(x, "x", torch.bfloat16, dev, 2)
    _need(codes, "codes", torch.uint8, dev, 2)
    _need(scales, "scales", torch.uint8, dev, 2)
    _need(s_g, "s_g", torch.float32, dev)
    M, d_o = g.shape
    d_i = x.shape[1]
    r = 0
    if A is not None or B is not None:
        _need(A, "A", torch.bfloat16, dev, 2)
        _need(B, "B", torch.bfloat16, dev, 2)
        r = A.shape[0]
    if w_norm is not None:
        _need(w_norm, "w_norm", torch.float32, dev, 1)
    z, z_ld = _noise(z, M, d_i, dev)
    dx = torch.empty(M, d_i, dtype=torch.float32, device=dev)
    dA = torch.empty(r, d_i, dtype=torch.float32, device=dev) if (r > 0 and want_adapter_grads) else None
    dB = torch.empty(d_o, r, dtype=torch.float32, device=dev) if (r > 0 and want_adapter_grads) else None
    need = int(lib().pl_backward_workspace_bytes(M, d_i, d_o, r, 1 if w_norm is not None else 0))
    if workspace is None:
        workspace = _default_ws.setdefault(dev, Workspace(dev))
    ws = workspace.get(max(need, 256))
    with torch.cuda.device(dev):
        st = lib().pl_nvfp4_lora_linear_backward(_ptr(g), M, d_i, d_o, _ptr(codes), _ptr(scales), _ptr(s_g), _ptr(A),
                                                 _ptr(B), r, float(lam), _ptr(x), _ptr(w_norm), _ptr(z), z_ld,
                                                 float(eps), _ptr(dx), _ptr(dA), _ptr(dB), _ptr(ws), ws.numel(),
                                                 _stream(dev))
    _check(st, "pl_nvfp4_lora_linear_backward")
    return dx, dA, dB


def aqn_stage(done: int, total: int) -> int:
    """Schedule stage (0 .. 9) after `done` of `total` planned updates."""
    k = int(lib().pl_aqn_stage(int(done), int(total)))
    if k < 0:
        raise ValueError("pl_aqn_stage: need total >= 1 and done >= 0")
    return k


def aqn_sigma(stage: int, sigma_start: float, sigma_end: float) -> float:
    """sigma of schedule stage `stage` (0 for the warm-up stage)."""
    v = float(lib().pl_aqn_sigma(int(stage), float(sigma_start), float(sigma_end)))
    if v < 0:
        raise ValueError("pl_aqn_sigma: stage outside 0..9 or non-positive endpoints")
    return v


def aqn_noise(d: int, seed: int, norm_id: int = 0, scope0: int = 0, n_scopes: int = 1, sigma: float = 1.0,
              out: torch.Tensor | None = None, device=None) -> torch.Tensor:
    """z FP32 [n_scopes, d]: the AQN noise states of scope indices scope0 .. scope0 + n_scopes - 1
    of norm `norm_id` under `seed` (row 0 is the z the linear and the norm take)."""
    dev = torch.device(device) if device is not None else (out.device if out is not None else torch.device("cuda"))
    if dev.type == "cuda" and dev.index is None:
        dev = torch.device("cuda", torch.cuda.current_device())
    if out is None:
        out = torch.empty(n_scopes, d, dtype=torch.float32, device=dev)
    _need(out, "out", torch.float32, dev, 2)
    if tuple(out.shape) != (n_scopes, d):
        raise ValueError(f"out must be [{n_scopes}, {d}]")
    with torch.cuda.device(dev):
        st = lib().pl_aqn_noise(int(seed) & 0xFFFFFFFFFFFFFFFF, int(norm_id) & 0xFFFFFFFF,
                                int(scope0) & 0xFFFFFFFFFFFFFFFF, int(n_scopes), int(d), float(sigma), _ptr(out),
                                _stream(dev))
    _check(st, "pl_aqn_noise")
    return out


def last_device_status(device=None) -> int:
    dev = torch.device(device) if device is not None else torch.device("cuda")
    with torch.cuda.device(dev):
        return int(lib().pl_last_device_status(_stream(dev)))


def linear_path(M: int, d_i: int, d_o: int, r: int) -> int:
    """Kernel path the linear takes for this shape on the current device: 2 fused
    tcgen05 kernel, 1 tcgen05 prologue + main kernel, 3 large-M CTA-pair contraction,
    0 CUDA-core kernels, -1 invalid."""
    return int(lib().pl_debug_linear_path(M, d_i, d_o, r))
