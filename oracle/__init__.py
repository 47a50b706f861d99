"""Plain CPU oracle for the multi-LoRA shrink / expand / expand_slice path.

TEST INFRASTRUCTURE ONLY.  The tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package; the product (the
CUDA library under ``lora_gemv_gb300`` and its binding) never does, and this
package imports nothing from the product.

The arithmetic lives in ``lora_oracle.c`` (double-precision loops over
tokens, see the comments there for the page each definition follows).  This
module only marshals numpy arrays to it.  All floating inputs are widened to
float64 before the call (fp16 / bf16 / fp32 widen exactly), so the oracle
sees exactly the values the GPU sees.

Parity pins: every function here is pinned by the CPU tests in
``tests/test_oracle_pins.py`` (closed forms, a library matmul special case,
a masked-sum reformulation, BGMV == SGMV, slices == concatenation,
rank-aware == zero-padded, library-sort grouping and a golden grouping from
Punica issue #17).  No function is left unpinned.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "lora_oracle.c")
# A prebuilt library may be named by LORA_ORACLE_LIB (the mutation tests load
# deliberately broken copies of the oracle this way); it is used as is.
_LIB = os.environ.get("LORA_ORACLE_LIB") or os.path.join(_HERE, "liblora_oracle.so")
_lib = None

TILE_DEFAULT = 64


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (plain -O2, no fast-math: IEEE double)."""
    if os.environ.get("LORA_ORACLE_LIB"):
        return _LIB
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
               "-fno-fast-math", "-ffp-contract=off", _SRC, "-o", tmp]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        i32p = ctypes.POINTER(ctypes.c_int32)
        f64p = ctypes.POINTER(ctypes.c_double)
        lib.oracle_num_threads.restype = ctypes.c_int
        lib.oracle_set_threads.argtypes = [ctypes.c_int]
        lib.oracle_map_tokens.argtypes = [i32p, ctypes.c_int32, ctypes.c_int32, i32p]
        lib.oracle_map_tokens.restype = ctypes.c_int
        lib.oracle_map_segments.argtypes = [i32p, i32p, i32p, ctypes.c_int32, ctypes.c_int32,
                                            ctypes.c_int32, i32p, i32p]
        lib.oracle_map_segments.restype = ctypes.c_int
        lib.oracle_group.argtypes = [i32p, ctypes.c_int32, ctypes.c_int32, ctypes.c_int,
                                     ctypes.c_int32, i32p, i32p, i32p, i32p, i32p, i32p,
                                     i32p, i32p]
        lib.oracle_group.restype = ctypes.c_int
        lib.oracle_shrink.argtypes = [f64p, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32,
                                      f64p, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                      i32p, i32p, ctypes.c_double, ctypes.c_int, f64p,
                                      ctypes.c_int64]
        lib.oracle_expand_slice.argtypes = [f64p, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32,
                                            ctypes.POINTER(f64p), i32p, i32p, ctypes.c_int32,
                                            ctypes.c_int32, ctypes.c_int32, i32p, i32p,
                                            ctypes.c_double, ctypes.c_int, f64p, ctypes.c_int64]
        _lib = lib
    return _lib


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _p(a: np.ndarray, ty):
    return a.ctypes.data_as(ctypes.POINTER(ty))


def num_threads() -> int:
    return _load().oracle_num_threads()


def set_threads(n: int) -> None:
    _load().oracle_set_threads(int(n))


def map_tokens(idx, L: int):
    """BGMV map: returns (lora_of[T] int32, bad_id_count)."""
    idx = _i32(idx)
    out = np.empty_like(idx)
    bad = _load().oracle_map_tokens(_p(idx, ctypes.c_int32), idx.size, int(L),
                                    _p(out, ctypes.c_int32))
    return out, bad


def map_segments(seg_start, seg_len, seg_lora, T: int, L: int):
    """SGMV map: returns (lora_of[T] int32, bad_id_count, error_bits)."""
    s, n, l = _i32(seg_start), _i32(seg_len), _i32(seg_lora)
    out = np.empty(int(T), dtype=np.int32)
    err = np.zeros(1, dtype=np.int32)
    bad = _load().oracle_map_segments(_p(s, ctypes.c_int32), _p(n, ctypes.c_int32),
                                      _p(l, ctypes.c_int32), s.size, int(T), int(L),
                                      _p(out, ctypes.c_int32), _p(err, ctypes.c_int32))
    return out, bad, int(err[0])


def group(lora_of, L: int, by_adapter: bool, tile: int = TILE_DEFAULT) -> dict:
    """Token grouping and tile list (see ``oracle_group`` in the C file)."""
    lo = _i32(lora_of)
    T = lo.size
    perm = np.empty(T, np.int32)
    count = np.empty(max(L, 1), np.int32)
    offset = np.empty(L + 1, np.int32)
    gl = np.empty(T + 1, np.int32)
    gs = np.empty(T + 1, np.int32)
    gc = np.empty(T + 1, np.int32)
    ng = np.zeros(1, np.int32)
    tiles = np.empty(4 * (T // max(tile, 1) + T + 2), np.int32)
    nt = _load().oracle_group(_p(lo, ctypes.c_int32), T, int(L), int(bool(by_adapter)),
                              int(tile), _p(perm, ctypes.c_int32), _p(count, ctypes.c_int32),
                              _p(offset, ctypes.c_int32), _p(gl, ctypes.c_int32),
                              _p(gs, ctypes.c_int32), _p(gc, ctypes.c_int32),
                              _p(ng, ctypes.c_int32), _p(tiles, ctypes.c_int32))
    g = int(ng[0])
    return {
        "perm": perm, "count": count[:L], "offset": offset, "n_active": int(offset[L]),
        "group_lora": gl[:g].copy(), "group_start": gs[:g].copy(),
        "group_count": gc[:g].copy(), "tiles": tiles[:4 * nt].reshape(nt, 4).copy(),
    }


def shrink(x, A, lora_of, *, num_slices: int = 1, ranks=None, scale: float = 1.0,
           add: bool = False, y=None) -> np.ndarray:
    """y[T, S*R] (float64).  x: [T, H]; A: [L, S*R, H]; lora_of: [T]."""
    x = _f64(x)
    A = _f64(A)
    T, H = x.shape
    L, SR, H2 = A.shape
    assert H2 == H and SR % num_slices == 0
    R = SR // num_slices
    lo = _i32(lora_of)
    assert lo.size == T
    if y is None:
        y = np.zeros((T, SR), np.float64)
    else:
        y = _f64(y).copy()
    assert y.shape[0] == T and y.shape[1] >= SR
    rk = _i32(ranks) if ranks is not None else None
    _load().oracle_shrink(_p(x, ctypes.c_double), H, T, H, _p(A, ctypes.c_double), L, R,
                          int(num_slices),
                          _p(rk, ctypes.c_int32) if rk is not None else None,
                          _p(lo, ctypes.c_int32), float(scale), int(bool(add)),
                          _p(y, ctypes.c_double), y.shape[1])
    return y


def expand_slice(y, B_list: Sequence, offsets: Sequence[int], lora_of, out, *,
                 y_stride: int, ranks=None, scale: float = 1.0,
                 add: bool = True) -> np.ndarray:
    """out[T, N_total] (float64) after expanding every slice.

    y: [T, >= S*y_stride]; B_list[s]: [L, N_s, R]; offsets[s]: first out column.
    """
    y = _f64(y)
    T = y.shape[0]
    Bs = [_f64(b) for b in B_list]
    L, _, R = Bs[0].shape
    for b in Bs:
        assert b.shape[0] == L and b.shape[2] == R
    Ns = _i32([b.shape[1] for b in Bs])
    offs = _i32(offsets)
    out = _f64(out).copy()
    assert out.shape[0] == T
    for s in range(len(Bs)):
        assert offs[s] >= 0 and offs[s] + Ns[s] <= out.shape[1]
        assert s * y_stride + R <= y.shape[1]
    lo = _i32(lora_of)
    rk = _i32(ranks) if ranks is not None else None
    f64p = ctypes.POINTER(ctypes.c_double)
    ptrs = (f64p * len(Bs))(*[_p(b, ctypes.c_double) for b in Bs])
    _load().oracle_expand_slice(_p(y, ctypes.c_double), y.shape[1], T, len(Bs), ptrs,
                                _p(Ns, ctypes.c_int32), _p(offs, ctypes.c_int32),
                                int(y_stride), L, R,
                                _p(rk, ctypes.c_int32) if rk is not None else None,
                                _p(lo, ctypes.c_int32), float(scale), int(bool(add)),
                                _p(out, ctypes.c_double), out.shape[1])
    return out


def expand(y, B, lora_of, out, *, ranks=None, scale: float = 1.0, add: bool = True):
    """Single-slice expand: out[T, N] (float64)."""
    B = _f64(B)
    return expand_slice(y, [B], [0], lora_of, out, y_stride=0, ranks=ranks, scale=scale,
                        add=add)
