"""Seeded synthetic tensors drawn directly on the GPU (for workloads too large
to draw on the host).  Wraps synth/synth.cu (libsynth.so) through ctypes.
Holds none of the BitDelta arithmetic."""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import torch

from . import LAPLACE_B, SIGMA_BASE

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.cu")
_LIB = os.path.join(_HERE, "libsynth.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    with _lock:
        if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
            nvcc = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
            tmp = _LIB + f".tmp{os.getpid()}"
            subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3",
                            "-std=c++17", "-Xcompiler", "-fPIC", "-shared", _SRC, "-o", tmp],
                           check=True)
            os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        p, i64, u64 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_uint64
        lib.synth_normal_bf16.argtypes = [p, i64, u64, u64, ctypes.c_float, p]
        lib.synth_normal_bf16.restype = ctypes.c_int
        lib.synth_finetuned_bf16.argtypes = [p, p, i64, u64, u64, ctypes.c_float, p]
        lib.synth_finetuned_bf16.restype = ctypes.c_int
        _lib = lib
    return _lib


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def normal_bf16(shape, seed: int, stream: int, sigma: float = 1.0, device="cuda"):
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    rc = _load().synth_normal_bf16(ctypes.c_void_p(out.data_ptr()), out.numel(), seed, stream,
                                   sigma, _stream())
    if rc != 0:
        raise RuntimeError(f"synth_normal_bf16 failed: cuda error {rc}")
    return out


def finetuned_bf16(base: torch.Tensor, seed: int, stream: int, b: float = LAPLACE_B):
    out = torch.empty_like(base)
    rc = _load().synth_finetuned_bf16(ctypes.c_void_p(out.data_ptr()),
                                      ctypes.c_void_p(base.data_ptr()), base.numel(), seed,
                                      stream, b, _stream())
    if rc != 0:
        raise RuntimeError(f"synth_finetuned_bf16 failed: cuda error {rc}")
    return out


def layer(seed: int, d_out: int, d_in: int, sigma: float = SIGMA_BASE, b: float = LAPLACE_B,
          stream: int = 0):
    """(W_base, W_ft) bf16 CUDA tensors [d_out, d_in]."""
    wb = normal_bf16((d_out, d_in), seed, 2 * stream + 1, sigma)
    return wb, finetuned_bf16(wb, seed, 2 * stream + 2, b)
