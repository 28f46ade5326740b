"""The C ABI without a GPU: the library loads, exports every symbol the header
declares, reports sizes, and rejects bad arguments on the host before launching."""

import ctypes
import os
import re

import pytest
import torch

from tests.conftest import ROOT

HEADER = os.path.join(ROOT, "include", "precision_linear.h")


@pytest.fixture(scope="module")
def L():
    from precision_linear_gb300 import binding, build
    build.build()
    return binding.lib()


def declared_functions():
    src = open(HEADER, encoding="utf-8").read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(pl_[a-z0-9_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(L):
    names = declared_functions()
    assert len(names) >= 9
    for n in names:
        assert hasattr(L, n), n


def test_status_strings_and_version(L):
    for s in range(11):
        txt = L.pl_status_string(s).decode()
        assert txt.startswith("PL_")
    assert L.pl_status_string(99).decode() == "unknown pl_status"
    assert L.pl_version() == 200


def test_nvfp4_bytes_is_9P_over_16(L):
    for d_o, d_i in [(256, 256), (3584, 3584), (512, 3584), (3584, 18944), (5120, 27648)]:
        assert L.pl_nvfp4_bytes(d_o, d_i) == 9 * d_o * d_i // 16
    assert L.pl_nvfp4_bytes(16, 24) == 0 and L.pl_nvfp4_bytes(0, 16) == 0


def test_workspace_bytes(L):
    assert L.pl_workspace_bytes(4, 256, 256, 8) > 0
    assert L.pl_workspace_bytes(64, 3584, 3584, 32) >= 64 * 3584 * 2
    assert L.pl_workspace_bytes(0, 256, 256, 8) == 0
    assert L.pl_workspace_bytes(4, 250, 256, 8) == 0
    assert L.pl_workspace_bytes(4, 256, 256, 65) == 0


FAKE = 1 << 20  # an aligned, never-dereferenced address


def _p(v):
    return ctypes.c_void_p(v)


def test_quantize_argument_checks(L):
    ok = (_p(FAKE), 16, 32, _p(FAKE), _p(FAKE), _p(FAKE), None)
    assert L.pl_nvfp4_quantize(None, *ok[1:]) == 1  # NULL
    assert L.pl_nvfp4_quantize(_p(FAKE), 16, 24, *ok[3:]) == 2  # d_i % 16
    assert L.pl_nvfp4_quantize(_p(FAKE), 0, 32, *ok[3:]) == 2
    assert L.pl_nvfp4_quantize(_p(FAKE + 8), *ok[1:]) == 3  # misaligned W


def test_rmsnorm_argument_checks(L):
    args = [_p(FAKE), 4, 256, _p(FAKE), None, 0, ctypes.c_float(1e-6), _p(FAKE), 0, None]
    a = list(args); a[0] = None
    assert L.pl_rmsnorm_aqn(*a) == 1
    a = list(args); a[2] = 250
    assert L.pl_rmsnorm_aqn(*a) == 2
    a = list(args); a[7] = _p(FAKE + 2)
    assert L.pl_rmsnorm_aqn(*a) == 3
    a = list(args); a[8] = 2  # not a pl_dtype
    assert L.pl_rmsnorm_aqn(*a) == 2
    # per-row noise: the row stride must be 0 or a multiple of 4 that is >= d
    for z_ld in (128, 258, -256):
        a = list(args); a[4] = _p(FAKE); a[5] = z_ld
        assert L.pl_rmsnorm_aqn(*a) == 2, z_ld
    a = list(args); a[4] = _p(FAKE + 4); a[5] = 256
    assert L.pl_rmsnorm_aqn(*a) == 3  # z rows must start 16-byte aligned


def _lin_args(**kw):
    d = dict(x=FAKE, M=4, d_i=256, d_o=256, codes=FAKE, scales=FAKE, s_g=FAKE, A=FAKE, B=FAKE, r=8,
             lam=2.0, w_norm=FAKE, z=FAKE, z_ld=0, eps=1e-6, y=FAKE, y_dtype=0, ws=FAKE, ws_bytes=1 << 30,
             stream=None)
    d.update(kw)
    return [_p(d["x"]) if d["x"] else None, d["M"], d["d_i"], d["d_o"], _p(d["codes"]) if d["codes"] else None,
            _p(d["scales"]), _p(d["s_g"]), _p(d["A"]) if d["A"] else None, _p(d["B"]) if d["B"] else None,
            d["r"], ctypes.c_float(d["lam"]), _p(d["w_norm"]) if d["w_norm"] else None,
            _p(d["z"]) if d["z"] else None, d["z_ld"], ctypes.c_float(d["eps"]), _p(d["y"]), d["y_dtype"],
            _p(d["ws"]) if d["ws"] else None, d["ws_bytes"], d["stream"]]


def test_linear_argument_checks(L):
    f = L.pl_nvfp4_lora_linear
    assert f(*_lin_args(x=0)) == 1
    assert f(*_lin_args(codes=0)) == 1
    assert f(*_lin_args(M=0)) == 2
    assert f(*_lin_args(d_i=250)) == 2
    assert f(*_lin_args(d_o=0)) == 2
    assert f(*_lin_args(r=65)) == 4
    assert f(*_lin_args(r=-1)) == 4
    assert f(*_lin_args(B=0)) == 1  # A without B
    assert f(*_lin_args(x=FAKE + 4)) == 3
    assert f(*_lin_args(ws=0)) == 7
    assert f(*_lin_args(ws_bytes=16)) == 7
    assert f(*_lin_args(ws=FAKE + 16)) == 7  # workspace must be 256-byte aligned
    assert f(*_lin_args(y_dtype=5)) == 2
    assert f(*_lin_args(z_ld=100)) == 2  # per-row noise rows shorter than d_i
    assert f(*_lin_args(z_ld=258)) == 2  # row stride not a multiple of 4
    assert f(*_lin_args(z_ld=-256)) == 2


def test_aqn_stage_and_sigma_follow_the_oracle(L):
    """Host-side schedule of the AQN noise against oracle/aqn.py (FP64, rounded to FP32)."""
    import numpy as np

    from oracle import aqn
    for total in (1, 7, 10, 1000, 12345):
        for done in sorted({0, 1, total // 10, total // 10 + 1, total // 2, total - 1, total, 3 * total}):
            assert L.pl_aqn_stage(done, total) == aqn.stage(done, total), (done, total)
    assert L.pl_aqn_stage(1 << 62, (1 << 62) + 1) == 9  # no overflow in 10 * done
    assert L.pl_aqn_stage(1, 0) == -1 and L.pl_aqn_stage(-1, 10) == -1
    for start, end in ((0.01, 0.0005), (0.05, 0.0005)):
        s32, e32 = float(np.float32(start)), float(np.float32(end))
        for k in range(10):
            want = np.float32(aqn.sigma(k, s32, e32))
            got = np.float32(L.pl_aqn_sigma(k, s32, e32))
            assert abs(int(got.view(np.int32)) - int(want.view(np.int32))) <= 1, (k, got, want)
        assert L.pl_aqn_sigma(1, s32, e32) == s32 and L.pl_aqn_sigma(9, s32, e32) == e32
    assert L.pl_aqn_sigma(10, 0.01, 0.0005) == -1.0 and L.pl_aqn_sigma(-1, 0.01, 0.0005) == -1.0
    assert L.pl_aqn_sigma(3, 0.0, 0.0005) == -1.0 and L.pl_aqn_sigma(3, 0.01, float("inf")) == -1.0


def test_uaq_argument_checks(L):
    q = L.pl_nvfp4_quantize_uaq
    ok = [_p(FAKE), 16, 32, ctypes.c_float(1.5), _p(FAKE), _p(FAKE), _p(FAKE), None]
    a = list(ok); a[0] = None
    assert q(*a) == 1
    for i, v in ((2, 24), (1, 0), (3, ctypes.c_float(0.0)), (3, ctypes.c_float(-1.5)),
                 (3, ctypes.c_float(float("inf")))):
        a = list(ok); a[i] = v
        assert q(*a) == 2, (i, v)
    a = list(ok); a[0] = _p(FAKE + 8)
    assert q(*a) == 3
    f = L.pl_uaq_fold_norm
    okf = [_p(FAKE), 256, ctypes.c_float(1.5), _p(FAKE), None]
    a = list(okf); a[3] = None
    assert f(*a) == 1
    a = list(okf); a[1] = 0
    assert f(*a) == 2
    a = list(okf); a[2] = ctypes.c_float(float("nan"))
    assert f(*a) == 2
    a = list(okf); a[0] = _p(FAKE + 2)
    assert f(*a) == 3


def test_aqn_noise_argument_checks(L):
    f = L.pl_aqn_noise
    ok = [1, 0, 0, 1, 256, ctypes.c_float(0.01), _p(FAKE), None]
    a = list(ok); a[6] = None
    assert f(*a) == 1
    for i, v in ((4, 0), (3, 0), (4, (1 << 31) + 1), (5, ctypes.c_float(-1.0)), (5, ctypes.c_float(float("nan")))):
        a = list(ok); a[i] = v
        assert f(*a) == 2, (i, v)
    a = list(ok); a[6] = _p(FAKE + 2)
    assert f(*a) == 3


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-device path")
def test_valid_arguments_without_a_device_report_device_error(L):
    assert L.pl_nvfp4_lora_linear(*_lin_args()) == 5
    assert L.pl_nvfp4_lora_linear(*_lin_args(z_ld=256)) == 5
    assert L.pl_rmsnorm_aqn(_p(FAKE), 4, 256, _p(FAKE), _p(FAKE), 256, ctypes.c_float(1e-6), _p(FAKE), 0, None) == 5
    assert L.pl_nvfp4_quantize(_p(FAKE), 16, 32, _p(FAKE), _p(FAKE), _p(FAKE), None) == 5
    assert L.pl_aqn_noise(1, 0, 0, 1, 256, ctypes.c_float(0.01), _p(FAKE), None) == 5
    assert L.pl_nvfp4_quantize_uaq(_p(FAKE), 16, 32, ctypes.c_float(1.5), _p(FAKE), _p(FAKE), _p(FAKE), None) == 5
    assert L.pl_uaq_fold_norm(_p(FAKE), 256, ctypes.c_float(1.5), _p(FAKE), None) == 5


def test_product_path_does_not_import_the_oracle():
    """The package and bench's product arm never reach oracle/: only tests, smoke()
    and the CPU-baseline legs may."""
    pkg = os.path.join(ROOT, "precision_linear_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                txt = open(os.path.join(dirpath, f), encoding="utf-8").read()
                assert not re.search(r"^\s*(from|import)\s+oracle\b", txt, re.M), f


def _proj_array(n, **kw):
    from precision_linear_gb300 import binding as pl
    arr = (pl.Proj * n)()
    for i in range(n):
        d = dict(d_o=256, codes=FAKE, scales=FAKE, s_g=FAKE, A=FAKE, B=FAKE, r=8, lam=2.0, y=FAKE)
        d.update(kw)
        arr[i] = pl.Proj(d["d_o"], d["codes"], d["scales"], d["s_g"], d["A"], d["B"], d["r"], d["lam"], d["y"])
    return arr


def test_group_argument_checks(L):
    from precision_linear_gb300 import binding as pl
    f = pl.lib().pl_nvfp4_lora_linear_group
    ok = lambda arr, n=None, **kw: [_p(kw.get("x", FAKE)) if kw.get("x", FAKE) else None, kw.get("M", 4), kw.get("d_i", 256),
                                    _p(FAKE), _p(FAKE), kw.get("z_ld", 0), ctypes.c_float(1e-6), arr,
                                    len(arr) if n is None else n, kw.get("y_dtype", 0),
                                    _p(kw.get("ws", FAKE)) if kw.get("ws", FAKE) else None, 1 << 30, None]
    assert f(*ok(_proj_array(2), x=0)) == 1
    assert f(*ok(_proj_array(2), n=0)) == 2
    assert f(*ok(_proj_array(9))) == 2           # more than PL_MAX_GROUP
    assert f(*ok(_proj_array(2), d_i=250)) == 2
    assert f(*ok(_proj_array(2), y_dtype=3)) == 2
    assert f(*ok(_proj_array(2), z_ld=100)) == 2
    assert f(*ok(_proj_array(2, r=65))) == 4
    assert f(*ok(_proj_array(2, codes=None))) == 1
    assert f(*ok(_proj_array(2, B=None))) == 1   # A without B
    assert f(*ok(_proj_array(2, y=FAKE + 8))) == 3
    assert f(*ok(_proj_array(2, d_o=0))) == 2
    assert f(*ok(_proj_array(2), ws=0)) == 7
    assert pl.lib().pl_workspace_bytes_group(4, 256, _proj_array(2), 2) > 0
    assert pl.lib().pl_workspace_bytes_group(4, 256, _proj_array(2), 0) == 0
    assert pl.lib().pl_workspace_bytes_group(4, 250, _proj_array(2), 2) == 0


def test_proj_struct_layout_matches_the_header(tmp_path):
    """The binding's ctypes mirror of pl_nvfp4_proj has the C compiler's size and offsets."""
    import shutil
    import subprocess
    from precision_linear_gb300 import binding as pl
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "layout.c"
    src.write_text('#include <stdio.h>\n#include <stddef.h>\n#include "precision_linear.h"\n'
                   'int main(void){printf("%zu %zu %zu %zu %zu\\n", sizeof(pl_nvfp4_proj), offsetof(pl_nvfp4_proj, r),'
                   ' offsetof(pl_nvfp4_proj, lambda), offsetof(pl_nvfp4_proj, y), offsetof(pl_nvfp4_proj, B_bf16));'
                   'return 0;}\n')
    exe = tmp_path / "layout"
    subprocess.check_call([cc, "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)])
    got = [int(v) for v in subprocess.check_output([str(exe)]).split()]
    P = pl.Proj
    assert got == [ctypes.sizeof(P), P.r.offset, P.lam.offset, P.y.offset, P.B.offset]


def test_w8a8_argument_checks(L):
    from precision_linear_gb300 import binding as pl
    q = pl.lib().pl_w8a8_quantize_weight
    assert q(None, 4, 32, _p(FAKE), _p(FAKE), None) == 1
    assert q(_p(FAKE), 4, 24, _p(FAKE), _p(FAKE), None) == 2
    assert q(_p(FAKE + 8), 4, 32, _p(FAKE), _p(FAKE), None) == 3
    f = pl.lib().pl_w8a8_lora_linear

    def args(**kw):
        d = dict(x=FAKE, M=4, d_i=256, d_o=64, codes=FAKE, s_w=FAKE, A=FAKE, B=FAKE, r=8, z_ld=0, y_dtype=0,
                 ws=FAKE, ws_bytes=1 << 30)
        d.update(kw)
        p = lambda v: _p(v) if v else None
        return [p(d["x"]), d["M"], d["d_i"], d["d_o"], p(d["codes"]), p(d["s_w"]), p(d["A"]), p(d["B"]), d["r"],
                ctypes.c_float(2.0), _p(FAKE), _p(FAKE), d["z_ld"], ctypes.c_float(1e-6), _p(FAKE), d["y_dtype"],
                p(d["ws"]), d["ws_bytes"], None]
    assert f(*args(x=0)) == 1
    assert f(*args(d_i=192)) == 2      # d_i % 128
    assert f(*args(d_i=64)) == 2
    assert f(*args(M=0)) == 2
    assert f(*args(r=65)) == 4
    assert f(*args(B=0)) == 1
    assert f(*args(ws=0)) == 7
    assert f(*args(ws_bytes=16)) == 7
    assert f(*args(z_ld=7)) == 2
    assert f(*args(x=FAKE + 4)) == 3
    assert pl.lib().pl_w8a8_workspace_bytes(4, 256, 64, 8) > 0
    assert pl.lib().pl_w8a8_workspace_bytes(4, 200, 64, 8) == 0


def test_backward_argument_checks(L):
    from precision_linear_gb300 import binding as pl
    f = pl.lib().pl_nvfp4_lora_linear_backward

    def args(**kw):
        d = dict(g=FAKE, M=4, d_i=256, d_o=64, A=FAKE, B=FAKE, r=8, x=FAKE, dx=FAKE, ws=FAKE, z_ld=0)
        d.update(kw)
        p = lambda v: _p(v) if v else None
        return [p(d["g"]), d["M"], d["d_i"], d["d_o"], _p(FAKE), _p(FAKE), _p(FAKE), p(d["A"]), p(d["B"]), d["r"],
                ctypes.c_float(2.0), p(d["x"]), _p(FAKE), _p(FAKE), d["z_ld"], ctypes.c_float(1e-6), p(d["dx"]),
                _p(FAKE), _p(FAKE), p(d["ws"]), 1 << 30, None]
    assert f(*args(g=0)) == 1
    assert f(*args(x=0)) == 1
    assert f(*args(dx=0)) == 1
    assert f(*args(d_i=128)) == 2    # d_i >= 256
    assert f(*args(d_i=384)) == 2    # d_i % 256 (the rows of block scales feed TMA)
    assert f(*args(d_o=60)) == 2     # d_o % 8
    assert f(*args(r=65)) == 4
    assert f(*args(B=0)) == 1
    assert f(*args(ws=0)) == 7
    assert f(*args(z_ld=3)) == 2
    assert f(*args(g=FAKE + 8)) == 3
    assert pl.lib().pl_backward_workspace_bytes(4, 256, 64, 8, 1) > pl.lib().pl_backward_workspace_bytes(4, 256, 64, 8, 0)
    assert pl.lib().pl_backward_workspace_bytes(4, 250, 64, 8, 1) == 0


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-device path")
def test_static_workspace_entry_reports_an_unsupported_device(L):
    from precision_linear_gb300 import binding as pl
    f = pl.lib().pl_nvfp4_lora_linear_static_ws
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p,
                  ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_void_p,
                  ctypes.c_void_p, ctypes.c_float, ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p]
    # a valid problem on a host without a device of compute capability 10.3: the device error,
    # not a failed symbol lookup
    st = f(_p(FAKE), 4, 256, 256, _p(FAKE), _p(FAKE), _p(FAKE), _p(FAKE), _p(FAKE), 8, ctypes.c_float(2.0), _p(FAKE),
           _p(FAKE), ctypes.c_float(1e-6), _p(FAKE), 0, None)
    assert st == 5


def _calls(n, over=None):
    from precision_linear_gb300 import binding as pl
    arr = (pl.Call * n)()
    for i in range(n):
        d = dict(x=FAKE + i * (1 << 16), M=4, d_o=256, codes=FAKE, scales=FAKE, s_g=FAKE, A=FAKE, B=FAKE, r=8,
                 lam=2.0, w_norm=FAKE, z=None, z_ld=0, y=FAKE + (1 << 24) + i * (1 << 16))
        d.update((over or {}).get(i, {}))
        arr[i] = pl.Call(d["x"], d["M"], d["d_o"], d["codes"], d["scales"], d["s_g"], d["A"], d["B"], d["r"],
                         d["lam"], d["w_norm"], d["z"], d["z_ld"], d["y"])
    return arr


def test_batch_argument_checks(L):
    from precision_linear_gb300 import binding as pl
    f = pl.lib().pl_nvfp4_lora_linear_batch
    ws = _p(FAKE)
    assert f(256, ctypes.c_float(1e-6), None, 2, 0, ws, 1 << 30, None) == 1
    assert f(256, ctypes.c_float(1e-6), _calls(2), 0, 0, ws, 1 << 30, None) == 2
    assert f(256, ctypes.c_float(1e-6), _calls(9), 9, 0, ws, 1 << 30, None) == 2  # more than PL_MAX_BATCH
    assert f(250, ctypes.c_float(1e-6), _calls(2), 2, 0, ws, 1 << 30, None) == 2
    assert f(256, ctypes.c_float(1e-6), _calls(2, {1: dict(x=None)}), 2, 0, ws, 1 << 30, None) == 1
    assert f(256, ctypes.c_float(1e-6), _calls(2, {1: dict(r=65)}), 2, 0, ws, 1 << 30, None) == 4
    assert f(256, ctypes.c_float(1e-6), _calls(2, {1: dict(y=FAKE + 8)}), 2, 0, ws, 1 << 30, None) == 3
    # an output overlapping another call's output, or any call's input: refused
    same_y = {1: dict(y=FAKE + (1 << 24))}
    assert f(256, ctypes.c_float(1e-6), _calls(2, same_y), 2, 0, ws, 1 << 30, None) == 10
    y_on_x = {0: dict(y=FAKE + (1 << 16) + 256)}
    assert f(256, ctypes.c_float(1e-6), _calls(2, y_on_x), 2, 0, ws, 1 << 30, None) == 10
    assert f(256, ctypes.c_float(1e-6), _calls(2), 2, 0, None, 1 << 30, None) == 7
    assert pl.lib().pl_workspace_bytes_batch(256, _calls(3), 3) > 0
    assert pl.lib().pl_workspace_bytes_batch(250, _calls(3), 3) == 0


def test_call_struct_layout_matches_the_header(tmp_path):
    import shutil
    import subprocess
    from precision_linear_gb300 import binding as pl
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "layout.c"
    src.write_text('#include <stdio.h>\n#include <stddef.h>\n#include "precision_linear.h"\n'
                   'int main(void){printf("%zu %zu %zu %zu %zu\\n", sizeof(pl_nvfp4_call), offsetof(pl_nvfp4_call, r),'
                   ' offsetof(pl_nvfp4_call, lambda), offsetof(pl_nvfp4_call, z_ld), offsetof(pl_nvfp4_call, y));'
                   'return 0;}\n')
    exe = tmp_path / "layout"
    subprocess.check_call([cc, "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)])
    got = [int(v) for v in subprocess.check_output([str(exe)]).split()]
    C = pl.Call
    assert got == [ctypes.sizeof(C), C.r.offset, C.lam.offset, C.z_ld.offset, C.y.offset]


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-device path")
def test_batch_without_a_device_reports_device_error(L):
    from precision_linear_gb300 import binding as pl
    assert pl.lib().pl_nvfp4_lora_linear_batch(256, ctypes.c_float(1e-6), _calls(3), 3, 0, _p(FAKE), 1 << 30,
                                               None) == 5
