"""Python binding of the GB300 multi-LoRA shrink / expand library.

Argument marshalling only: every step of the path runs in the CUDA kernels of
``liblora_gemv.so`` (C ABI in ``include/lora_gemv.h``).  PyTorch supplies
device memory and the current stream.  There is no CPU fallback: if the
library is missing or a tensor is not on a CUDA device, the call raises.

Functions carry the C names:

* ``lora_workspace_size(T, L)`` / ``lora_plan_layout(T, L)``
* ``lora_group_tokens(token_idx, L, plan)``                 BGMV plan
* ``lora_group_segments(seg_start, seg_len, seg_lora, T, L, plan)``  SGMV plan
* ``lora_shrink(x, A, y, plan, ...)``
* ``lora_expand(y, B, out, plan, ...)``
* ``lora_expand_slice(y, B_slices, out, plan, slice_offsets, ...)``
* ``lora_shrink_expand_slice(x, A, y, B_slices, out, plan, slice_offsets, ...)``
* ``lora_bgmv_shrink(x, A, y, token_idx, ...)``, ``lora_bgmv_expand_slice(y, B_slices, out,
  slice_offsets, token_idx, ...)``, ``lora_bgmv_shrink_expand_slice(...)``: the plan-free
  decode path (token_idx None = one adapter for every token)
* ``lora_shrink_expand_slice_noalloc(token_idx, x, A, y, B_slices, out, slice_offsets, ...)``
  (the decode pair with the library's own plan array: no plan argument)
* ``lora_get_error(plan)``
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "liblora_gemv.so")
DEBUG_LIB_PATH = os.path.join(_HERE, "liblora_gemv_debug.so")  # the LORA_DEBUG build

LORA_F16, LORA_BF16 = 0, 1
TILE_TOKENS = 64
MAX_RANK = 128
MAX_SLICES = 8
HDR_WORDS = 16
HDR = dict(MAGIC=0, T=1, L=2, KIND=3, NACTIVE=4, NGROUPS=5, NTILES=6, BAD_IDS=7, ERR=8)
PLANERR_SEG_RANGE, PLANERR_SEG_ORDER, PLANERR_MISMATCH, PLANERR_TIMEOUT = 1, 2, 4, 8
PLANERR_BOUNDS = 16
PLAN_MAGIC = 0x4C6F5241

EXPORTS = ("lora_plan_layout", "lora_workspace_size", "lora_group_tokens",
           "lora_group_segments", "lora_shrink", "lora_expand", "lora_expand_slice",
           "lora_shrink_expand_slice", "lora_shrink_expand_slice_noalloc", "lora_get_error",
           "lora_status_string", "lora_last_error_detail", "lora_version", "lora_bgmv_shrink",
           "lora_bgmv_expand_slice", "lora_bgmv_shrink_expand_slice",
           "lora_bgmv_fused_shrink_expand_slice")
NOALLOC_MAX_TOKENS = 4096
BGMV_MAX_ADAPTERS = 8
FUSED_MAX_TOKENS = 256

_lib = None
_lib_path = None


class LoraError(RuntimeError):
    def __init__(self, status: int, detail: str):
        super().__init__(f"lora status {status}: {detail}")
        self.status = status


class _Layout(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int64) for n in ("header", "count", "offset", "perm", "group_lora",
                                             "group_start", "group_count", "tiles", "tile_rows",
                                             "max_tiles", "bytes")]


def use_library(path: Optional[str] = None) -> None:
    """Route every following call through the library at `path` (None: the
    default build, LIB_PATH).  The LORA_DEBUG variant is DEBUG_LIB_PATH."""
    global _lib, _lib_path
    _lib_path = path or LIB_PATH
    _lib = None


def load():
    """Load the CUDA library (raises if it was not built)."""
    global _lib
    if _lib is not None:
        return _lib
    path = _lib_path or LIB_PATH
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with lora_gemv_gb300.build.build() "
                           "(there is no CPU fallback)")
    lib = ctypes.CDLL(path)
    vp, i32, i64, f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float
    st = ctypes.c_int
    lib.lora_plan_layout.argtypes = [i32, i32, ctypes.POINTER(_Layout)]
    lib.lora_plan_layout.restype = st
    lib.lora_workspace_size.argtypes = [i32, i32]
    lib.lora_workspace_size.restype = ctypes.c_size_t
    lib.lora_group_tokens.argtypes = [vp, i32, i32, vp, ctypes.c_size_t, vp]
    lib.lora_group_tokens.restype = st
    lib.lora_group_segments.argtypes = [vp, vp, vp, i32, i32, i32, vp, ctypes.c_size_t, vp]
    lib.lora_group_segments.restype = st
    lib.lora_shrink.argtypes = [st, vp, i64, i32, i32, vp, i32, i32, i32, vp, vp, i64, vp, f32,
                                ctypes.c_int, vp]
    lib.lora_shrink.restype = st
    lib.lora_expand.argtypes = [st, vp, i64, i32, vp, i32, i32, i32, vp, vp, i64, vp, f32,
                                ctypes.c_int, vp]
    lib.lora_expand.restype = st
    lib.lora_expand_slice.argtypes = [st, vp, i64, i32, i32, ctypes.POINTER(vp),
                                      ctypes.POINTER(i32), ctypes.POINTER(i32), i32, i32, i32, vp,
                                      vp, i64, vp, f32, ctypes.c_int, vp]
    lib.lora_expand_slice.restype = st
    lib.lora_shrink_expand_slice.argtypes = [st, vp, i64, i32, i32, vp, i32, i32, vp, vp, i64, i32,
                                             ctypes.POINTER(vp), ctypes.POINTER(i32),
                                             ctypes.POINTER(i32), vp, i64, vp, f32, f32,
                                             ctypes.c_int, vp]
    lib.lora_shrink_expand_slice.restype = st
    lib.lora_shrink_expand_slice_noalloc.argtypes = [st, vp, vp, i64, i32, i32, vp, i32, i32, vp,
                                                     vp, i64, i32, ctypes.POINTER(vp),
                                                     ctypes.POINTER(i32), ctypes.POINTER(i32), vp,
                                                     i64, f32, f32, ctypes.c_int, vp]
    lib.lora_shrink_expand_slice_noalloc.restype = st
    lib.lora_bgmv_shrink.argtypes = [st, vp, vp, i64, i32, i32, vp, i32, i32, i32, vp, vp, i64,
                                     f32, ctypes.c_int, vp, vp]
    lib.lora_bgmv_shrink.restype = st
    lib.lora_bgmv_expand_slice.argtypes = [st, vp, vp, i64, i32, i32, ctypes.POINTER(vp),
                                           ctypes.POINTER(i32), ctypes.POINTER(i32), i32, i32, i32,
                                           vp, vp, i64, f32, ctypes.c_int, vp, vp]
    lib.lora_bgmv_expand_slice.restype = st
    lib.lora_bgmv_shrink_expand_slice.argtypes = [st, vp, vp, i64, i32, i32, vp, i32, i32, vp, vp,
                                                  i64, i32, ctypes.POINTER(vp),
                                                  ctypes.POINTER(i32), ctypes.POINTER(i32), vp,
                                                  i64, f32, f32, ctypes.c_int, vp, vp]
    lib.lora_bgmv_shrink_expand_slice.restype = st
    lib.lora_bgmv_fused_shrink_expand_slice.argtypes = [st, vp, vp, i64, i32, i32, vp, i32, i32, vp,
                                                        vp, i64, i32, ctypes.POINTER(vp),
                                                        ctypes.POINTER(i32), ctypes.POINTER(i32),
                                                        vp, i64, f32, f32, ctypes.c_int, vp]
    lib.lora_bgmv_fused_shrink_expand_slice.restype = st
    lib.lora_get_error.argtypes = [vp, ctypes.POINTER(i32), ctypes.POINTER(i32), vp]
    lib.lora_get_error.restype = st
    lib.lora_status_string.argtypes = [st]
    lib.lora_status_string.restype = ctypes.c_char_p
    lib.lora_last_error_detail.restype = ctypes.c_char_p
    lib.lora_version.restype = i32
    _lib = lib
    return lib


def _check(status: int) -> None:
    if status != 0:
        lib = load()
        raise LoraError(status, f"{lib.lora_status_string(status).decode()}: "
                                f"{lib.lora_last_error_detail().decode()}")


def _stream(t: torch.Tensor) -> int:
    return torch.cuda.current_stream(t.device).cuda_stream


def _dev(t: torch.Tensor, name: str) -> int:
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (there is no CPU path)")
    return t.data_ptr()


def _dtype(t: torch.Tensor) -> int:
    if t.dtype == torch.float16:
        return LORA_F16
    if t.dtype == torch.bfloat16:
        return LORA_BF16
    raise ValueError(f"unsupported dtype {t.dtype}: fp16 or bf16")


def _rows(t: torch.Tensor, name: str) -> int:
    """Leading dimension of a row-major 2-D tensor with unit inner stride."""
    if t.dim() != 2 or (t.stride(1) != 1 and t.shape[1] > 1):
        raise ValueError(f"{name} must be 2-D with unit column stride")
    return t.stride(0) if t.shape[0] > 1 else max(t.shape[1], 1)


def _i32(t: Optional[torch.Tensor], name: str) -> Optional[int]:
    if t is None:
        return None
    if t.dtype != torch.int32 or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous int32 tensor")
    return _dev(t, name)


# ------------------------------------------------------------------ plan

def lora_plan_layout(T: int, L: int) -> dict:
    lay = _Layout()
    _check(load().lora_plan_layout(int(T), int(L), ctypes.byref(lay)))
    return {n: getattr(lay, n) for n, _ in _Layout._fields_}


def lora_workspace_size(T: int, L: int) -> int:
    return int(load().lora_workspace_size(int(T), int(L)))


def new_plan(T: int, L: int, device="cuda") -> torch.Tensor:
    """A plan buffer (uint8 device tensor, 16-byte aligned by the allocator)."""
    n = lora_workspace_size(T, L)
    if n == 0:
        _check(load().lora_plan_layout(int(T), int(L), ctypes.byref(_Layout())))
    return torch.empty(n, dtype=torch.uint8, device=device)


def lora_group_tokens(token_idx: torch.Tensor, L: int, plan: torch.Tensor) -> None:
    T = token_idx.numel()
    _check(load().lora_group_tokens(_i32(token_idx, "token_idx"), T, int(L),
                                    _dev(plan, "plan"), plan.numel() * plan.element_size(),
                                    _stream(plan)))


def lora_group_segments(seg_start: torch.Tensor, seg_len: torch.Tensor, seg_lora: torch.Tensor,
                        T: int, L: int, plan: torch.Tensor) -> None:
    S = seg_start.numel()
    if seg_len.numel() != S or seg_lora.numel() != S:
        raise ValueError("segment arrays differ in length")
    _check(load().lora_group_segments(_i32(seg_start, "seg_start"), _i32(seg_len, "seg_len"),
                                      _i32(seg_lora, "seg_lora"), S, int(T), int(L),
                                      _dev(plan, "plan"), plan.numel() * plan.element_size(),
                                      _stream(plan)))


def plan_view(plan: torch.Tensor, T: int, L: int) -> dict:
    """Device views of the plan arrays (int32), for inspection and tests."""
    lay = lora_plan_layout(T, L)
    w = plan.view(torch.int32)

    def seg(off, n):
        return w[off // 4: off // 4 + n]

    return {
        "header": seg(lay["header"], HDR_WORDS),
        "count": seg(lay["count"], L),
        "offset": seg(lay["offset"], L + 1),
        "perm": seg(lay["perm"], T),
        "group_lora": seg(lay["group_lora"], T + 1),
        "group_start": seg(lay["group_start"], T + 1),
        "group_count": seg(lay["group_count"], T + 1),
        "tiles": seg(lay["tiles"], 4 * lay["max_tiles"]).view(-1, 4),
        "tile_rows": seg(lay["tile_rows"], TILE_TOKENS * lay["max_tiles"]).view(-1, TILE_TOKENS),
    }


def lora_get_error(plan: torch.Tensor):
    """(bad_ids, err_flags) of a plan; synchronises the current stream."""
    bad, err = ctypes.c_int32(), ctypes.c_int32()
    _check(load().lora_get_error(_dev(plan, "plan"), ctypes.byref(bad), ctypes.byref(err),
                                 _stream(plan)))
    return bad.value, err.value


# ------------------------------------------------------------------ operators

def lora_shrink(x: torch.Tensor, A: torch.Tensor, y: torch.Tensor, plan: torch.Tensor, *,
                num_slices: int = 1, ranks: Optional[torch.Tensor] = None, scale: float = 1.0,
                add_inputs: bool = False) -> None:
    """y[:, :S*R] (+)= scale * x @ A[idx]^T (rank-aware).  x [T, H], A [L, S*R, H]
    contiguous, y [T, >= S*R] fp32 with unit column stride."""
    T, H = x.shape
    if A.dim() != 3 or not A.is_contiguous() or A.shape[2] != H or A.dtype != x.dtype:
        raise ValueError("A must be a contiguous [L, S*R, H] tensor of x's dtype")
    L, SR, _ = A.shape
    if SR % num_slices:
        raise ValueError("A rows are not a multiple of num_slices")
    if y.dtype != torch.float32 or y.shape[0] != T or y.shape[1] < SR:
        raise ValueError("y must be fp32 [T, >= S*R]")
    _check(load().lora_shrink(_dtype(x), _dev(x, "x"), _rows(x, "x"), T, H, _dev(A, "A"), L,
                              SR // num_slices, num_slices, _i32(ranks, "ranks"), _dev(y, "y"),
                              _rows(y, "y"), _dev(plan, "plan"), float(scale),
                              int(bool(add_inputs)), _stream(x)))


def lora_expand(y: torch.Tensor, B: torch.Tensor, out: torch.Tensor, plan: torch.Tensor, *,
                ranks: Optional[torch.Tensor] = None, scale: float = 1.0,
                add_inputs: bool = True) -> None:
    """out[:, :N] (+)= scale * y[:, :R] @ B[idx]^T.  B [L, N, R] contiguous."""
    if B.dim() != 3 or not B.is_contiguous() or B.dtype != out.dtype:
        raise ValueError("B must be a contiguous [L, N, R] tensor of out's dtype")
    L, N, R = B.shape
    T = out.shape[0]
    if y.dtype != torch.float32 or y.shape[0] != T or y.shape[1] < R:
        raise ValueError("y must be fp32 [T, >= R]")
    if out.shape[1] < N:
        raise ValueError("out has fewer than N columns")
    _check(load().lora_expand(_dtype(out), _dev(y, "y"), _rows(y, "y"), T, _dev(B, "B"), L, N,
                              R, _i32(ranks, "ranks"), _dev(out, "out"), _rows(out, "out"),
                              _dev(plan, "plan"), float(scale), int(bool(add_inputs)),
                              _stream(out)))


def lora_expand_slice(y: torch.Tensor, B_slices: Sequence[torch.Tensor], out: torch.Tensor,
                      plan: torch.Tensor, slice_offsets: Sequence[int], *, y_slice_stride: int,
                      ranks: Optional[torch.Tensor] = None, scale: float = 1.0,
                      add_inputs: bool = True) -> None:
    """Every slice s: out[:, off_s:off_s+N_s] (+)= scale * y[:, s*ys : s*ys+R] @ B_s[idx]^T,
    all slices in one launch.  B_s [L, N_s, R] contiguous."""
    S = len(B_slices)
    if S != len(slice_offsets):
        raise ValueError("one offset per slice")
    L, _, R = B_slices[0].shape
    for b in B_slices:
        if b.dim() != 3 or not b.is_contiguous() or b.shape[0] != L or b.shape[2] != R \
                or b.dtype != out.dtype:
            raise ValueError("every B_s must be a contiguous [L, N_s, R] tensor of out's dtype")
    T = out.shape[0]
    if y.dtype != torch.float32 or y.shape[0] != T \
            or y.shape[1] < (S - 1) * int(y_slice_stride) + R:
        raise ValueError("y must be fp32 [T, >= (S-1)*y_slice_stride + R]")
    if any(int(o) + b.shape[1] > out.shape[1] for o, b in zip(slice_offsets, B_slices)):
        raise ValueError("a slice ends past out's columns")
    ptrs = (ctypes.c_void_p * S)(*[_dev(b, "B_s") for b in B_slices])
    Ns = (ctypes.c_int32 * S)(*[b.shape[1] for b in B_slices])
    offs = (ctypes.c_int32 * S)(*[int(o) for o in slice_offsets])
    _check(load().lora_expand_slice(_dtype(out), _dev(y, "y"), _rows(y, "y"), T, S, ptrs, Ns,
                                    offs, int(y_slice_stride), L, R, _i32(ranks, "ranks"),
                                    _dev(out, "out"), _rows(out, "out"), _dev(plan, "plan"),
                                    float(scale), int(bool(add_inputs)), _stream(out)))


def lora_shrink_expand_slice(x: torch.Tensor, A: torch.Tensor, y: torch.Tensor,
                             B_slices: Sequence[torch.Tensor], out: torch.Tensor,
                             plan: torch.Tensor, slice_offsets: Sequence[int], *,
                             ranks: Optional[torch.Tensor] = None, scale_shrink: float = 1.0,
                             scale_expand: float = 1.0, add_inputs: bool = True) -> None:
    """y = scale_shrink * x @ A[idx]^T (written), then every slice s:
    out[:, off_s:off_s+N_s] (+)= scale_expand * y[:, s*R:(s+1)*R] @ B_s[idx]^T.
    A [L, S*R, H], B_s [L, N_s, R] contiguous; S = len(B_slices)."""
    T, H = x.shape
    S = len(B_slices)
    if A.dim() != 3 or not A.is_contiguous() or A.shape[2] != H or A.dtype != x.dtype:
        raise ValueError("A must be a contiguous [L, S*R, H] tensor of x's dtype")
    L, SR, _ = A.shape
    if SR % S or S != len(slice_offsets):
        raise ValueError("A rows must be S*R with one offset per slice")
    R = SR // S
    for b in B_slices:
        if b.dim() != 3 or not b.is_contiguous() or b.shape[0] != L or b.shape[2] != R \
                or b.dtype != out.dtype or out.dtype != x.dtype:
            raise ValueError("every B_s must be a contiguous [L, N_s, R] tensor of x's dtype")
    if y.dtype != torch.float32 or y.shape[0] != T or y.shape[1] < SR:
        raise ValueError("y must be fp32 [T, >= S*R]")
    if out.shape[0] != T or any(int(o) + b.shape[1] > out.shape[1]
                                for o, b in zip(slice_offsets, B_slices)):
        raise ValueError("a slice ends past out's columns")
    ptrs = (ctypes.c_void_p * S)(*[_dev(b, "B_s") for b in B_slices])
    Ns = (ctypes.c_int32 * S)(*[b.shape[1] for b in B_slices])
    offs = (ctypes.c_int32 * S)(*[int(o) for o in slice_offsets])
    _check(load().lora_shrink_expand_slice(
        _dtype(x), _dev(x, "x"), _rows(x, "x"), T, H, _dev(A, "A"), L, R, _i32(ranks, "ranks"),
        _dev(y, "y"), _rows(y, "y"), S, ptrs, Ns, offs, _dev(out, "out"), _rows(out, "out"),
        _dev(plan, "plan"), float(scale_shrink), float(scale_expand), int(bool(add_inputs)),
        _stream(x)))


def lora_shrink_expand_slice_noalloc(token_idx: torch.Tensor, x: torch.Tensor, A: torch.Tensor,
                                     y: torch.Tensor, B_slices: Sequence[torch.Tensor],
                                     out: torch.Tensor, slice_offsets: Sequence[int], *,
                                     ranks: Optional[torch.Tensor] = None,
                                     scale_shrink: float = 1.0, scale_expand: float = 1.0,
                                     add_inputs: bool = True) -> None:
    """As lora_group_tokens followed by lora_shrink_expand_slice, with the plan
    kept in the library's own device array (no plan buffer; T <= 4096; calls
    on one device must not overlap on the GPU)."""
    T, H = x.shape
    S = len(B_slices)
    if A.dim() != 3 or not A.is_contiguous() or A.shape[2] != H or A.dtype != x.dtype:
        raise ValueError("A must be a contiguous [L, S*R, H] tensor of x's dtype")
    L, SR, _ = A.shape
    if SR % S or S != len(slice_offsets):
        raise ValueError("A rows must be S*R with one offset per slice")
    if token_idx.numel() != T:
        raise ValueError("token_idx must hold one index per row of x")
    R = SR // S
    for b in B_slices:
        if b.dim() != 3 or not b.is_contiguous() or b.shape[0] != L or b.shape[2] != R \
                or b.dtype != out.dtype or out.dtype != x.dtype:
            raise ValueError("every B_s must be a contiguous [L, N_s, R] tensor of x's dtype")
    if y.dtype != torch.float32 or y.shape[0] != T or y.shape[1] < SR:
        raise ValueError("y must be fp32 [T, >= S*R]")
    if out.shape[0] != T or any(int(o) + b.shape[1] > out.shape[1]
                                for o, b in zip(slice_offsets, B_slices)):
        raise ValueError("a slice ends past out's columns")
    ptrs = (ctypes.c_void_p * S)(*[_dev(b, "B_s") for b in B_slices])
    Ns = (ctypes.c_int32 * S)(*[b.shape[1] for b in B_slices])
    offs = (ctypes.c_int32 * S)(*[int(o) for o in slice_offsets])
    _check(load().lora_shrink_expand_slice_noalloc(
        _dtype(x), _i32(token_idx, "token_idx"), _dev(x, "x"), _rows(x, "x"), T, H, _dev(A, "A"),
        L, R, _i32(ranks, "ranks"), _dev(y, "y"), _rows(y, "y"), S, ptrs, Ns, offs,
        _dev(out, "out"), _rows(out, "out"), float(scale_shrink), float(scale_expand),
        int(bool(add_inputs)), _stream(x)))


# ------------------------------------------------------------------ plan-free BGMV

def _slices(B_slices, slice_offsets, out, L, R):
    S = len(B_slices)
    if S != len(slice_offsets):
        raise ValueError("one offset per slice")
    for b in B_slices:
        if b.dim() != 3 or not b.is_contiguous() or b.shape[0] != L or b.shape[2] != R \
                or b.dtype != out.dtype:
            raise ValueError("every B_s must be a contiguous [L, N_s, R] tensor of out's dtype")
    if any(int(o) + b.shape[1] > out.shape[1] for o, b in zip(slice_offsets, B_slices)):
        raise ValueError("a slice ends past out's columns")
    ptrs = (ctypes.c_void_p * S)(*[_dev(b, "B_s") for b in B_slices])
    Ns = (ctypes.c_int32 * S)(*[b.shape[1] for b in B_slices])
    offs = (ctypes.c_int32 * S)(*[int(o) for o in slice_offsets])
    return S, ptrs, Ns, offs


def lora_bgmv_shrink(x: torch.Tensor, A: torch.Tensor, y: torch.Tensor,
                     token_idx: Optional[torch.Tensor], *, num_slices: int = 1,
                     ranks: Optional[torch.Tensor] = None, scale: float = 1.0,
                     add_inputs: bool = False, status: Optional[torch.Tensor] = None) -> None:
    """Plan-free y[:, :S*R] (+)= scale * x @ A[idx]^T.  token_idx [T] int32 or None
    (every token uses adapter 0); status: optional int32 device word."""
    T, H = x.shape
    if A.dim() != 3 or not A.is_contiguous() or A.shape[2] != H or A.dtype != x.dtype:
        raise ValueError("A must be a contiguous [L, S*R, H] tensor of x's dtype")
    L, SR, _ = A.shape
    if SR % num_slices:
        raise ValueError("A rows are not a multiple of num_slices")
    if y.dtype != torch.float32 or y.shape[0] != T or y.shape[1] < SR:
        raise ValueError("y must be fp32 [T, >= S*R]")
    if token_idx is not None and token_idx.numel() != T:
        raise ValueError("token_idx must hold one index per row of x")
    _check(load().lora_bgmv_shrink(_dtype(x), _i32(token_idx, "token_idx"), _dev(x, "x"),
                                   _rows(x, "x"), T, H, _dev(A, "A"), L, SR // num_slices,
                                   num_slices, _i32(ranks, "ranks"), _dev(y, "y"), _rows(y, "y"),
                                   float(scale), int(bool(add_inputs)), _i32(status, "status"),
                                   _stream(x)))


def lora_bgmv_expand_slice(y: torch.Tensor, B_slices: Sequence[torch.Tensor], out: torch.Tensor,
                           slice_offsets: Sequence[int], token_idx: Optional[torch.Tensor], *,
                           y_slice_stride: int, ranks: Optional[torch.Tensor] = None,
                           scale: float = 1.0, add_inputs: bool = True,
                           status: Optional[torch.Tensor] = None) -> None:
    """Plan-free expand_slice: every slice s, out[:, off_s:off_s+N_s] (+)=
    scale * y[:, s*ys : s*ys+R] @ B_s[idx]^T, all slices in one launch."""
    L, _, R = B_slices[0].shape
    T = out.shape[0]
    S, ptrs, Ns, offs = _slices(B_slices, slice_offsets, out, L, R)
    if y.dtype != torch.float32 or y.shape[0] != T \
            or y.shape[1] < (S - 1) * int(y_slice_stride) + R:
        raise ValueError("y must be fp32 [T, >= (S-1)*y_slice_stride + R]")
    if token_idx is not None and token_idx.numel() != T:
        raise ValueError("token_idx must hold one index per row of out")
    _check(load().lora_bgmv_expand_slice(_dtype(out), _i32(token_idx, "token_idx"), _dev(y, "y"),
                                         _rows(y, "y"), T, S, ptrs, Ns, offs,
                                         int(y_slice_stride), L, R, _i32(ranks, "ranks"),
                                         _dev(out, "out"), _rows(out, "out"), float(scale),
                                         int(bool(add_inputs)), _i32(status, "status"),
                                         _stream(out)))


def lora_bgmv_shrink_expand_slice(x: torch.Tensor, A: torch.Tensor, y: torch.Tensor,
                                  B_slices: Sequence[torch.Tensor], out: torch.Tensor,
                                  slice_offsets: Sequence[int],
                                  token_idx: Optional[torch.Tensor], *,
                                  ranks: Optional[torch.Tensor] = None,
                                  scale_shrink: float = 1.0, scale_expand: float = 1.0,
                                  add_inputs: bool = True,
                                  status: Optional[torch.Tensor] = None) -> None:
    """Plan-free shrink then expand_slice (y_slice_stride = R), chained."""
    T, H, L, R, S, ptrs, Ns, offs = _pair_args(x, A, y, B_slices, out, slice_offsets, token_idx)
    _check(load().lora_bgmv_shrink_expand_slice(
        _dtype(x), _i32(token_idx, "token_idx"), _dev(x, "x"), _rows(x, "x"), T, H, _dev(A, "A"),
        L, R, _i32(ranks, "ranks"), _dev(y, "y"), _rows(y, "y"), S, ptrs, Ns, offs,
        _dev(out, "out"), _rows(out, "out"), float(scale_shrink), float(scale_expand),
        int(bool(add_inputs)), _i32(status, "status"), _stream(x)))


def lora_bgmv_fused_shrink_expand_slice(x: torch.Tensor, A: torch.Tensor, y: torch.Tensor,
                                        B_slices: Sequence[torch.Tensor], out: torch.Tensor,
                                        slice_offsets: Sequence[int],
                                        token_idx: Optional[torch.Tensor], *,
                                        ranks: Optional[torch.Tensor] = None,
                                        scale_shrink: float = 1.0, scale_expand: float = 1.0,
                                        add_inputs: bool = True) -> None:
    """lora_bgmv_shrink_expand_slice as one cooperative kernel launch
    (T <= FUSED_MAX_TOKENS, R <= 32)."""
    T, H, L, R, S, ptrs, Ns, offs = _pair_args(x, A, y, B_slices, out, slice_offsets, token_idx)
    _check(load().lora_bgmv_fused_shrink_expand_slice(
        _dtype(x), _i32(token_idx, "token_idx"), _dev(x, "x"), _rows(x, "x"), T, H, _dev(A, "A"),
        L, R, _i32(ranks, "ranks"), _dev(y, "y"), _rows(y, "y"), S, ptrs, Ns, offs,
        _dev(out, "out"), _rows(out, "out"), float(scale_shrink), float(scale_expand),
        int(bool(add_inputs)), _stream(x)))


def _pair_args(x, A, y, B_slices, out, slice_offsets, token_idx):
    T, H = x.shape
    if A.dim() != 3 or not A.is_contiguous() or A.shape[2] != H or A.dtype != x.dtype:
        raise ValueError("A must be a contiguous [L, S*R, H] tensor of x's dtype")
    L, SR, _ = A.shape
    S = len(B_slices)
    if SR % S:
        raise ValueError("A rows must be S*R")
    R = SR // S
    if out.dtype != x.dtype or out.shape[0] != T:
        raise ValueError("out must be [T, N_total] of x's dtype")
    S, ptrs, Ns, offs = _slices(B_slices, slice_offsets, out, L, R)
    if y.dtype != torch.float32 or y.shape[0] != T or y.shape[1] < SR:
        raise ValueError("y must be fp32 [T, >= S*R]")
    if token_idx is not None and token_idx.numel() != T:
        raise ValueError("token_idx must hold one index per row of x")
    return T, H, L, R, S, ptrs, Ns, offs
