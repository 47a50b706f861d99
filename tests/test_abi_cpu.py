"""CPU-side checks of the C ABI: the library builds and loads, exports every
function include/lora_gemv.h declares, and rejects bad arguments on the host
before touching the GPU (no compute call is made here)."""
import ctypes
import os
import re

import pytest

import lora_gemv_gb300 as lg
from lora_gemv_gb300 import build as lgbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    lgbuild.build()
    return lg.load()


def declared_functions():
    names = set()
    for f in os.listdir(os.path.join(ROOT, "include")):
        if f.endswith(".h"):
            text = open(os.path.join(ROOT, "include", f)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"\b(lora_\w+)\s*\(", text))
    return names


def test_exports_every_declared_function(lib):
    names = declared_functions()
    assert {"lora_shrink", "lora_expand", "lora_expand_slice", "lora_group_tokens",
            "lora_group_segments", "lora_get_error"} <= names
    for n in names:
        assert hasattr(lib, n), n
    assert set(lg.EXPORTS) == names


def test_debug_build_exports_every_declared_function():
    """The LORA_DEBUG variant builds (cross-compiled here) and exports the
    same C ABI."""
    path = lgbuild.build(debug=True)
    assert path.endswith("liblora_gemv_debug.so") and os.path.exists(path)
    dlib = ctypes.CDLL(path)
    for n in declared_functions():
        assert hasattr(dlib, n), n


def test_version_and_status_strings(lib):
    assert lib.lora_version() == 100
    for s in range(5):
        assert lib.lora_status_string(s)
    assert lib.lora_status_string(99) == b"unknown status"


def test_plan_layout(lib):
    lay = lg.lora_plan_layout(1000, 4)
    assert lay["header"] == 0 and lay["count"] == 64
    assert lay["offset"] == 64 + 16 and lay["perm"] == 64 + 16 + 20
    assert lay["tiles"] % 16 == 0
    assert lay["max_tiles"] == 1000 + 1000 // 64 + 2
    assert lay["tile_rows"] == lay["tiles"] + 16 * lay["max_tiles"]
    assert lay["bytes"] == lay["tile_rows"] + 4 * 64 * lay["max_tiles"]
    assert lg.lora_workspace_size(1000, 4) == lay["bytes"]
    assert lg.lora_workspace_size(-1, 4) == 0
    assert lg.lora_workspace_size(10, 0) == 0
    assert lg.lora_workspace_size(10, 2000) == 0
    with pytest.raises(lg.LoraError):
        lg.lora_plan_layout(10, 0)


def test_host_validation_before_any_launch(lib):
    """Bad arguments are rejected on the host (no CUDA call is reached)."""
    vp = ctypes.c_void_p
    fake = vp(0x10000)  # never dereferenced: validation fails first
    # bad dtype
    assert lib.lora_shrink(7, fake, 64, 4, 64, fake, 2, 16, 1, None, fake, 16, fake, 1.0, 0,
                           None) == 1
    # R out of range
    assert lib.lora_shrink(0, fake, 64, 4, 64, fake, 2, 129, 1, None, fake, 129, fake, 1.0, 0,
                           None) == 1
    # ldx < H
    assert lib.lora_shrink(0, fake, 32, 4, 64, fake, 2, 16, 1, None, fake, 16, fake, 1.0, 0,
                           None) == 1
    # ldy < S*R
    assert lib.lora_shrink(0, fake, 64, 4, 64, fake, 2, 16, 2, None, fake, 16, fake, 1.0, 0,
                           None) == 1
    # plan misaligned
    assert lib.lora_shrink(0, fake, 64, 4, 64, fake, 2, 16, 1, None, fake, 16, vp(0x10004), 1.0,
                           0, None) == 3
    # group_tokens: plan too small, L too large
    assert lib.lora_group_tokens(fake, 100, 4, fake, 10, None) == 3
    assert lib.lora_group_tokens(fake, 100, 5000, fake, 1 << 30, None) == 2
    assert b"L = 5000" in lib.lora_last_error_detail()
    # expand_slice: overlapping slices, slice past ldo, too many slices
    S = 2
    Bs = (vp * S)(fake, fake)
    Ns = (ctypes.c_int32 * S)(32, 32)
    ov = (ctypes.c_int32 * S)(0, 16)
    assert lib.lora_expand_slice(0, fake, 16, 4, S, Bs, Ns, ov, 0, 2, 16, None, fake, 64, fake,
                                 1.0, 1, None) == 1
    past = (ctypes.c_int32 * S)(0, 40)
    assert lib.lora_expand_slice(0, fake, 16, 4, S, Bs, Ns, past, 0, 2, 16, None, fake, 64, fake,
                                 1.0, 1, None) == 1
    ok = (ctypes.c_int32 * S)(0, 32)
    assert lib.lora_expand_slice(0, fake, 16, 4, 9, Bs, Ns, ok, 0, 2, 16, None, fake, 64, fake,
                                 1.0, 1, None) == 1
    # y columns of the last slice beyond ldy
    assert lib.lora_expand_slice(0, fake, 16, 4, S, Bs, Ns, ok, 16, 2, 16, None, fake, 64, fake,
                                 1.0, 1, None) == 1
    # get_error on NULL
    assert lib.lora_get_error(None, None, None, None) == 1


def test_binding_refuses_cpu_tensors(lib):
    import torch
    with pytest.raises(ValueError):
        lg.lora_group_tokens(torch.zeros(4, dtype=torch.int32), 2, torch.zeros(4096,
                                                                                dtype=torch.uint8))
