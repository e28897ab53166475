"""Plain CPU oracle of the BitDelta hot path (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` import this package.  It wraps ``oracle/oracle.cpp`` (a
single-threaded fp64 C++ implementation written from the page "BitDelta:
serving 14 Zen models from one GPU cluster") through ctypes on numpy host
arrays.  It shares no code with the CUDA library and never touches a GPU.

All bf16 tensors are passed as ``numpy.uint16`` bit patterns.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.cpp")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

# -ffp-contract=off: no fused multiply-add, every operation rounds once.
_CXXFLAGS = ["-O2", "-std=c++17", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math"]


def build(force: bool = False) -> str:
    """Compile liboracle.so next to its source if it is missing or stale."""
    with _lock:
        stale = (not os.path.exists(_LIB_PATH)) or (
            os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
        if force or stale:
            tmp = _LIB_PATH + f".tmp{os.getpid()}"
            subprocess.run(["g++", *_CXXFLAGS, _SRC, "-o", tmp], check=True)
            os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        i64, i32, p = ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p
        lib.orc_packed_bytes.argtypes = [i64, i64]
        lib.orc_packed_bytes.restype = i64
        lib.orc_bf16_round.argtypes = [ctypes.c_float]
        lib.orc_bf16_round.restype = ctypes.c_uint16
        lib.orc_compress.argtypes = [p, p, i64, i64, ctypes.c_int, p, p, p]
        lib.orc_compress.restype = None
        lib.orc_reconstruct.argtypes = [p, p, p, ctypes.c_int, i64, i64, p]
        lib.orc_reconstruct.restype = None
        lib.orc_linear.argtypes = [p, i64, p, p, p, ctypes.c_int, i64, i64, p]
        lib.orc_linear.restype = None
        lib.orc_linear_split.argtypes = [p, i64, p, p, p, ctypes.c_int, i64, i64, p]
        lib.orc_linear_split.restype = None
        lib.orc_linear_at.argtypes = [p, i64, p, p, p, ctypes.c_int, i64, i64, p, p, i64, p]
        lib.orc_linear_at.restype = None
        lib.orc_linear_grouped.argtypes = [p, i64, p, p, i32, p, p, p, i32, ctypes.c_int,
                                           i64, i64, p]
        lib.orc_linear_grouped.restype = None
        lib.orc_linear_grouped_at.argtypes = [p, i64, p, p, i32, p, p, p, i32, ctypes.c_int,
                                              i64, i64, p, p, i64, p]
        lib.orc_linear_grouped_at.restype = None
        lib.orc_sign_cosine.argtypes = [p, p, p, p, ctypes.c_int, i64, i64, p]
        lib.orc_sign_cosine.restype = None
        _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def packed_bytes(d_out: int, d_in: int) -> int:
    return int(_load().orc_packed_bytes(d_out, d_in))


def bf16_round(f: float) -> int:
    return int(_load().orc_bf16_round(ctypes.c_float(f)))


def compress(w_base, w_ft, per_row: bool):
    """Return (packed uint8 [d_out, d_in/8], alpha float32, alpha float64)."""
    wb = _c(w_base, np.uint16)
    wf = _c(w_ft, np.uint16)
    d_out, d_in = wb.shape
    assert wf.shape == wb.shape and d_in % 8 == 0
    packed = np.empty((d_out, d_in // 8), np.uint8)
    n_alpha = d_out if per_row else 1
    a32 = np.empty(n_alpha, np.float32)
    a64 = np.empty(n_alpha, np.float64)
    _load().orc_compress(_ptr(wb), _ptr(wf), d_out, d_in, int(per_row), _ptr(packed),
                         _ptr(a32), _ptr(a64))
    return packed, a32, a64


def reconstruct(w_base, packed, alpha, per_row: bool):
    wb = _c(w_base, np.uint16)
    pk = _c(packed, np.uint8)
    al = _c(alpha, np.float32)
    d_out, d_in = wb.shape
    out = np.empty_like(wb)
    _load().orc_reconstruct(_ptr(wb), _ptr(pk), _ptr(al), int(per_row), d_out, d_in, _ptr(out))
    return out


def linear(x, w_base, packed, alpha, per_row: bool):
    """fp64 y [M, d_out] = x · W_effᵀ."""
    xx = _c(x, np.uint16)
    wb = _c(w_base, np.uint16)
    pk = _c(packed, np.uint8)
    al = _c(alpha, np.float32)
    M = xx.shape[0]
    d_out, d_in = wb.shape
    y = np.empty((M, d_out), np.float64)
    _load().orc_linear(_ptr(xx), M, _ptr(wb), _ptr(pk), _ptr(al), int(per_row), d_out, d_in,
                       _ptr(y))
    return y


def linear_split(x, w_base, packed, alpha, per_row: bool):
    """fp64 y [M, d_out] = x·W_baseᵀ + α ⊙ (x·Sᵀ): the effective weight
    W_base + α·sign(Δ) as a real number, not rounded to bf16."""
    xx = _c(x, np.uint16)
    wb = _c(w_base, np.uint16)
    pk = _c(packed, np.uint8)
    al = _c(alpha, np.float32)
    M = xx.shape[0]
    d_out, d_in = wb.shape
    y = np.empty((M, d_out), np.float64)
    _load().orc_linear_split(_ptr(xx), M, _ptr(wb), _ptr(pk), _ptr(al), int(per_row), d_out, d_in,
                             _ptr(y))
    return y


def linear_at(x, w_base, packed, alpha, per_row: bool, m_idx, n_idx):
    """fp64 y[m_idx[i], n_idx[i]] for each sample i."""
    xx = _c(x, np.uint16)
    wb = _c(w_base, np.uint16)
    pk = _c(packed, np.uint8)
    al = _c(alpha, np.float32)
    mi = _c(m_idx, np.int64)
    ni = _c(n_idx, np.int64)
    d_out, d_in = wb.shape
    out = np.empty(mi.shape[0], np.float64)
    _load().orc_linear_at(_ptr(xx), xx.shape[0], _ptr(wb), _ptr(pk), _ptr(al), int(per_row),
                          d_out, d_in, _ptr(mi), _ptr(ni), mi.shape[0], _ptr(out))
    return out


def _variant_tables(packed_list, alpha_list):
    pk = [_c(p, np.uint8) for p in packed_list]
    al = [_c(a, np.float32) for a in alpha_list]
    n_var = len(pk)
    pk_arr = (ctypes.c_void_p * max(n_var, 1))(*[p.ctypes.data for p in pk])
    al_arr = (ctypes.c_void_p * max(n_var, 1))(*[a.ctypes.data for a in al])
    return pk, al, pk_arr, al_arr, n_var


def linear_grouped(x, seg_offsets, seg_variant, w_base, packed_list, alpha_list, per_row: bool):
    xx = _c(x, np.uint16)
    so = _c(seg_offsets, np.int32)
    sv = _c(seg_variant, np.int32)
    wb = _c(w_base, np.uint16)
    keep = _variant_tables(packed_list, alpha_list)
    _, _, pk_arr, al_arr, n_var = keep
    d_out, d_in = wb.shape
    y = np.zeros((xx.shape[0], d_out), np.float64)
    _load().orc_linear_grouped(_ptr(xx), xx.shape[0], _ptr(so), _ptr(sv), sv.shape[0], _ptr(wb),
                               pk_arr, al_arr, n_var, int(per_row), d_out, d_in, _ptr(y))
    return y


def linear_grouped_at(x, seg_offsets, seg_variant, w_base, packed_list, alpha_list,
                      per_row: bool, m_idx, n_idx):
    xx = _c(x, np.uint16)
    so = _c(seg_offsets, np.int32)
    sv = _c(seg_variant, np.int32)
    wb = _c(w_base, np.uint16)
    keep = _variant_tables(packed_list, alpha_list)
    _, _, pk_arr, al_arr, n_var = keep
    mi = _c(m_idx, np.int64)
    ni = _c(n_idx, np.int64)
    d_out, d_in = wb.shape
    out = np.empty(mi.shape[0], np.float64)
    _load().orc_linear_grouped_at(_ptr(xx), xx.shape[0], _ptr(so), _ptr(sv), sv.shape[0],
                                  _ptr(wb), pk_arr, al_arr, n_var, int(per_row), d_out, d_in,
                                  _ptr(mi), _ptr(ni), mi.shape[0], _ptr(out))
    return out


def sign_cosine(packed_a, alpha_a, packed_b, alpha_b, per_row: bool):
    """[K-Merge] cosine of the task vectors α_a⊙S_a and α_b⊙S_b (1-bit form).
    Returns (cos, dot, |a|², |b|²), all fp64."""
    pa, pb = _c(packed_a, np.uint8), _c(packed_b, np.uint8)
    aa, ab = _c(alpha_a, np.float32), _c(alpha_b, np.float32)
    d_out, row_bytes = pa.shape
    out = np.zeros(4, np.float64)
    _load().orc_sign_cosine(_ptr(pa), _ptr(aa), _ptr(pb), _ptr(ab), int(per_row), d_out,
                            row_bytes * 8, _ptr(out))
    return tuple(float(v) for v in out)


def monosoup_merge(w_base, w_ft_list, rank: int):
    """[MonoSoup] W_base + (1/k)·Σ rank-r truncated SVD of each Δ_i.
    Returns (W_merged bf16 bits, W_merged fp64, correction fp64);
    see oracle/monosoup.py."""
    from . import monosoup as _ms
    return _ms.monosoup(_c(w_base, np.uint16), [_c(w, np.uint16) for w in w_ft_list], rank)
