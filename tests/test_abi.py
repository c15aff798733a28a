"""The C-ABI library: it builds for sm_103a, loads, exports exactly the functions
include/rec_attn.h declares, and rejects bad arguments on the host before any
CUDA call (so these checks need no GPU)."""
import ctypes
import os
import re

import numpy as np
import pytest

from generative_recommender_ranking_gb300 import binding as bd
from generative_recommender_ranking_gb300 import build as bld

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    bld.build()
    return bd.lib()


def _declared():
    with open(os.path.join(ROOT, "include", "rec_attn.h")) as f:
        src = f.read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(rec_attn_[a-z_]+)\s*\(", src)))


def test_exports_every_declared_symbol(L):
    names = _declared()
    assert {"rec_attn_plan", "rec_attn_fwd", "rec_attn_free"} <= set(names)
    for n in names:
        assert hasattr(L, n), n


def test_exports_nothing_else(L):
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", bd.library_path()], capture_output=True,
                         text=True, check=True).stdout
    exported = sorted({ln.split()[-1] for ln in out.splitlines()
                       if ln.split() and ln.split()[-1].startswith("rec_attn")})
    assert exported == _declared()


def test_status_strings(L):
    for code in range(7):
        s = bd.rec_attn_status_string(code)
        assert s and s != "unknown status"
    assert bd.rec_attn_status_string(99) == "unknown status"


def _plan_code(L, params, offsets, dev=1, out=True):
    off = np.asarray(offsets, dtype=np.int64)
    h = ctypes.c_void_p()
    return L.rec_attn_plan(ctypes.byref(params), len(off) - 1, off.ctypes.data, dev, dev, dev, None,
                           ctypes.byref(h) if out else None)


def test_host_validation_rejects_bad_arguments(L):
    good = bd.make_params(4, 64)
    off = [0, 100, 300]
    bad_abi = bd.make_params(4, 64); bad_abi.abi_version = 2
    assert _plan_code(L, bad_abi, off) == bd.ERR_INVALID_ARG
    assert _plan_code(L, bd.make_params(0, 64), off) == bd.ERR_INVALID_ARG
    assert _plan_code(L, bd.make_params(4, 63), off) == bd.ERR_INVALID_ARG
    assert _plan_code(L, bd.make_params(4, 96), off) == bd.ERR_UNSUPPORTED
    assert _plan_code(L, bd.make_params(4, 32), off) == bd.ERR_UNSUPPORTED          # bf16 needs 64/128
    assert _plan_code(L, bd.make_params(4, 128, dtype="fp32"), off) == bd.ERR_UNSUPPORTED
    assert _plan_code(L, bd.make_params(4, 64, window=-1), off) == bd.ERR_INVALID_ARG
    assert _plan_code(L, bd.make_params(4, 64, use_delay=True, delay_s=-5), off) == bd.ERR_INVALID_ARG
    assert _plan_code(L, bd.make_params(4, 64, dt_max_s=0.0), off) == bd.ERR_INVALID_ARG
    assert _plan_code(L, bd.make_params(4, 64, rope_base=float("nan")), off) == bd.ERR_INVALID_ARG
    assert _plan_code(L, bd.make_params(4, 64, softmax_scale=-1.0), off) == bd.ERR_INVALID_ARG
    p = bd.make_params(4, 64); p.use_rope = 2
    assert _plan_code(L, p, off) == bd.ERR_INVALID_ARG
    # offsets: must start at 0 and not decrease; lengths are capped
    assert _plan_code(L, good, [1, 100]) == bd.ERR_INVALID_ARG
    assert _plan_code(L, good, [0, 100, 50]) == bd.ERR_INVALID_ARG
    assert _plan_code(L, good, [0, bd.MAX_REQUEST_LEN + 1]) == bd.ERR_UNSUPPORTED
    assert _plan_code(L, good, [0, 2 ** 31]) == bd.ERR_UNSUPPORTED
    # NULL device arrays and NULL out pointer
    assert _plan_code(L, good, off, dev=None) == bd.ERR_INVALID_ARG
    assert _plan_code(L, good, off, out=False) == bd.ERR_INVALID_ARG
    h = ctypes.c_void_p()
    assert L.rec_attn_plan(None, 1, None, None, None, None, None, ctypes.byref(h)) == bd.ERR_INVALID_ARG
    assert L.rec_attn_plan(ctypes.byref(good), -1, None, None, None, None, None,
                           ctypes.byref(h)) == bd.ERR_INVALID_ARG
    assert h.value is None


def test_null_plan_calls(L):
    assert L.rec_attn_fwd(None, 1, 1, 1, 1, None, None) == bd.ERR_INVALID_ARG
    f = bd.RecAttnFused(None, None, 1e-6, None, None, None)
    assert L.rec_attn_fwd_fused(None, 1, 1, 1, ctypes.byref(f), 1, None, None) == bd.ERR_INVALID_ARG
    n = ctypes.c_size_t()
    assert L.rec_attn_tile_classes(None, None, 0, ctypes.byref(n)) == bd.ERR_INVALID_ARG
    c = ctypes.c_uint64()
    assert L.rec_attn_visible_pairs(None, ctypes.byref(c)) == bd.ERR_INVALID_ARG
    s = ctypes.c_int32()
    assert L.rec_attn_device_status(None, ctypes.byref(s)) == bd.ERR_INVALID_ARG
    L.rec_attn_free(None)  # NULL-safe
    st = ctypes.c_int32()
    assert L.rec_attn_check_wait_timeout(0, ctypes.byref(st), None) == bd.ERR_INVALID_ARG
    assert L.rec_attn_check_wait_timeout(20000, ctypes.byref(st), None) == bd.ERR_INVALID_ARG
    assert L.rec_attn_check_wait_timeout(50, None, None) == bd.ERR_INVALID_ARG


def test_valid_plan_without_gpu_reports_cuda_error(L):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert _plan_code(L, bd.make_params(4, 64), [0, 100, 300]) == bd.ERR_CUDA


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(bd, "_LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(bd, "_lib", None)
    with pytest.raises(OSError):
        bd.lib()
