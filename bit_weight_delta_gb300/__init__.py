"""Thin Python binding of libbitdelta.so (the GB300 BitDelta hot path).

Every function here only marshals arguments: it checks tensor devices and
dtypes, allocates outputs through torch (device memory is plumbing), and calls
the C entry point of the same name declared in include/bitdelta.h.  All
arithmetic runs in the library's CUDA kernels; there is no CPU or PyTorch
fallback.  If the library cannot be loaded, importing works but every call
raises.

bf16 tensors are torch.bfloat16; the packed sign matrix is torch.uint8
[d_out, d_in/8]; alpha is torch.float32 ([1] or [d_out]).
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import _build

PER_MATRIX = 0
PER_ROW = 1

_STATUS = {
    0: "BD_OK", 1: "BD_ERR_INVALID_ARG", 2: "BD_ERR_UNSUPPORTED_SHAPE", 3: "BD_ERR_MISALIGNED",
    4: "BD_ERR_WORKSPACE", 5: "BD_ERR_CUDA", 6: "BD_ERR_DEVICE_TIMEOUT",
    7: "BD_ERR_DEVICE_BOUNDS",
}

EXPORTED = (
    "bitdelta_packed_bytes", "bitdelta_compress_workspace_bytes", "bitdelta_compress",
    "bitdelta_reconstruct", "bitdelta_linear", "bitdelta_linear_grouped",
    "bitdelta_check_error", "bitdelta_set_wait_limit_ns", "bitdelta_debug_wait_timeout",
    "bitdelta_status_string", "bitdelta_compress_noalloc",
)


class BitDeltaError(RuntimeError):
    def __init__(self, fn: str, code: int):
        self.code = code
        super().__init__(f"{fn} failed: {_STATUS.get(code, code)} ({status_string(code)})")


_lib = None


def library_path() -> str:
    return _build.LIB_PATH


def load(build_if_missing: bool = True) -> ctypes.CDLL:
    """Load libbitdelta.so (building it in-tree first if it is missing or stale)."""
    global _lib
    if _lib is not None:
        return _lib
    if build_if_missing:
        _build.build()
    if not os.path.exists(_build.LIB_PATH):
        raise RuntimeError(f"libbitdelta.so not found at {_build.LIB_PATH}; run the build")
    lib = ctypes.CDLL(_build.LIB_PATH)
    i64, i32, p, sz = ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p, ctypes.c_size_t
    st = ctypes.c_int
    lib.bitdelta_packed_bytes.argtypes = [i64, i64]
    lib.bitdelta_packed_bytes.restype = sz
    lib.bitdelta_compress_workspace_bytes.argtypes = [i64, i64, st]
    lib.bitdelta_compress_workspace_bytes.restype = sz
    lib.bitdelta_compress.argtypes = [p, p, i64, i64, st, p, p, p, sz, p]
    lib.bitdelta_compress.restype = st
    lib.bitdelta_compress_noalloc.argtypes = [p, p, i64, i64, st, p, p, p]
    lib.bitdelta_compress_noalloc.restype = st
    lib.bitdelta_reconstruct.argtypes = [p, p, p, st, i64, i64, p, p]
    lib.bitdelta_reconstruct.restype = st
    lib.bitdelta_linear.argtypes = [p, i64, p, p, p, st, i64, i64, p, p]
    lib.bitdelta_linear.restype = st
    lib.bitdelta_linear_grouped.argtypes = [p, i64, p, p, i32, i32, p, p, p, i32, st, i64, i64,
                                            p, p]
    lib.bitdelta_linear_grouped.restype = st
    lib.bitdelta_check_error.argtypes = [p]
    lib.bitdelta_check_error.restype = st
    lib.bitdelta_set_wait_limit_ns.argtypes = [ctypes.c_uint64]
    lib.bitdelta_set_wait_limit_ns.restype = st
    lib.bitdelta_debug_wait_timeout.argtypes = [p]
    lib.bitdelta_debug_wait_timeout.restype = st
    lib.bitdelta_status_string.argtypes = [st]
    lib.bitdelta_status_string.restype = ctypes.c_char_p
    _lib = lib
    return lib


def status_string(code: int) -> str:
    return load().bitdelta_status_string(int(code)).decode()


def _check(fn: str, code: int) -> None:
    if code != 0:
        raise BitDeltaError(fn, code)


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _ptr(t: torch.Tensor | None) -> ctypes.c_void_p:
    return ctypes.c_void_p(0 if t is None else t.data_ptr())


def _dev(t: torch.Tensor, dtype, name: str) -> torch.Tensor:
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def _mode(per_row: bool) -> int:
    return PER_ROW if per_row else PER_MATRIX


def bitdelta_packed_bytes(d_out: int, d_in: int) -> int:
    return int(load().bitdelta_packed_bytes(d_out, d_in))


def bitdelta_compress_workspace_bytes(d_out: int, d_in: int, per_row: bool) -> int:
    return int(load().bitdelta_compress_workspace_bytes(d_out, d_in, _mode(per_row)))


def bitdelta_compress(w_base, w_ft, per_row: bool = True, packed_out=None, alpha_out=None,
                      workspace=None, stream=None):
    """Packed signs and α of Δ = W_ft − W_base.  Returns (packed, alpha)."""
    _dev(w_base, torch.bfloat16, "w_base")
    _dev(w_ft, torch.bfloat16, "w_ft")
    d_out, d_in = w_base.shape
    if packed_out is None:
        packed_out = torch.empty((d_out, d_in // 8), dtype=torch.uint8, device=w_base.device)
    if alpha_out is None:
        alpha_out = torch.empty((d_out if per_row else 1,), dtype=torch.float32,
                                device=w_base.device)
    need = bitdelta_compress_workspace_bytes(d_out, d_in, per_row)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=w_base.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("bitdelta_compress", load().bitdelta_compress(
        _ptr(w_base), _ptr(w_ft), d_out, d_in, _mode(per_row), _ptr(packed_out), _ptr(alpha_out),
        _ptr(workspace), ws_bytes, _stream(stream)))
    return packed_out, alpha_out


def bitdelta_compress_noalloc(w_base, w_ft, per_row: bool, packed_out, alpha_out, stream=None):
    """bitdelta_compress for callers that cannot allocate device memory: the
    outputs are passed in and the library allocates nothing (per-matrix α
    uses a fixed device array, d_out <= 65536).  Returns (packed, alpha)."""
    _dev(w_base, torch.bfloat16, "w_base")
    _dev(w_ft, torch.bfloat16, "w_ft")
    _dev(packed_out, torch.uint8, "packed_out")
    _dev(alpha_out, torch.float32, "alpha_out")
    d_out, d_in = w_base.shape
    _check("bitdelta_compress_noalloc", load().bitdelta_compress_noalloc(
        _ptr(w_base), _ptr(w_ft), d_out, d_in, _mode(per_row), _ptr(packed_out),
        _ptr(alpha_out), _stream(stream)))
    return packed_out, alpha_out


def bitdelta_reconstruct(w_base, packed, alpha, per_row: bool = True, out=None, stream=None):
    """W_eff = bf16(fp32(W_base) ± α) written to memory."""
    _dev(w_base, torch.bfloat16, "w_base")
    _dev(packed, torch.uint8, "packed")
    _dev(alpha, torch.float32, "alpha")
    d_out, d_in = w_base.shape
    if out is None:
        out = torch.empty_like(w_base)
    _check("bitdelta_reconstruct", load().bitdelta_reconstruct(
        _ptr(w_base), _ptr(packed), _ptr(alpha), _mode(per_row), d_out, d_in, _ptr(out),
        _stream(stream)))
    return out


def bitdelta_linear(x, w_base, packed, alpha, per_row: bool = True, out=None, stream=None):
    """y = x · (W_base + α·sign(Δ))ᵀ, x [..., d_in] bf16 -> y [..., d_out] bf16."""
    _dev(x, torch.bfloat16, "x")
    _dev(w_base, torch.bfloat16, "w_base")
    _dev(packed, torch.uint8, "packed")
    _dev(alpha, torch.float32, "alpha")
    d_out, d_in = w_base.shape
    lead = x.shape[:-1]
    M = x.numel() // d_in if x.numel() else 0
    if out is None:
        out = torch.empty((*lead, d_out), dtype=torch.bfloat16, device=x.device)
    _check("bitdelta_linear", load().bitdelta_linear(
        _ptr(x), M, _ptr(w_base), _ptr(packed), _ptr(alpha), _mode(per_row), d_out, d_in,
        _ptr(out), _stream(stream)))
    return out


def variant_tables(packed_list, alpha_list, device):
    """Device arrays of the variants' packed and α pointers (slot v-1 = variant v).

    The returned tensors must stay alive while the tables are used; the
    caller keeps them together with the listed tensors."""
    pk = torch.tensor([t.data_ptr() for t in packed_list] or [0], dtype=torch.int64,
                      device=device)
    al = torch.tensor([t.data_ptr() for t in alpha_list] or [0], dtype=torch.int64,
                      device=device)
    return pk, al


def bitdelta_linear_grouped(x, seg_offsets, seg_variant, w_base, packed_table, alpha_table,
                            n_var: int, max_seg_len: int, per_row: bool = True, out=None,
                            stream=None):
    """Multi-tenant linear: rows of segment s use variant seg_variant[s] (0 = base).

    seg_offsets int32 [n_seg+1] and seg_variant int32 [n_seg] are CUDA tensors;
    packed_table / alpha_table are int64 CUDA tensors of device pointers, as
    made by variant_tables()."""
    _dev(x, torch.bfloat16, "x")
    _dev(w_base, torch.bfloat16, "w_base")
    _dev(seg_offsets, torch.int32, "seg_offsets")
    _dev(seg_variant, torch.int32, "seg_variant")
    d_out, d_in = w_base.shape
    M = x.shape[0]
    if out is None:
        out = torch.empty((M, d_out), dtype=torch.bfloat16, device=x.device)
    _check("bitdelta_linear_grouped", load().bitdelta_linear_grouped(
        _ptr(x), M, _ptr(seg_offsets), _ptr(seg_variant), seg_variant.numel(), int(max_seg_len),
        _ptr(w_base), _ptr(packed_table), _ptr(alpha_table), int(n_var), _mode(per_row), d_out,
        d_in, _ptr(out), _stream(stream)))
    return out


def bitdelta_check_error(stream=None) -> int:
    """Synchronise and return (then clear) the device error status code."""
    return int(load().bitdelta_check_error(_stream(stream)))


def bitdelta_set_wait_limit_ns(ns: int) -> None:
    _check("bitdelta_set_wait_limit_ns", load().bitdelta_set_wait_limit_ns(int(ns)))


def bitdelta_debug_wait_timeout(stream=None) -> None:
    _check("bitdelta_debug_wait_timeout", load().bitdelta_debug_wait_timeout(_stream(stream)))
