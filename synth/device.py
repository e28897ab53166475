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


def finetuned_bf16(base: torch.Tensor, seed: int, stream: int, b: float = LAPLACE_B,
                   out: torch.Tensor = None):
    out = torch.empty_like(base) if out is None else out
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


# --------------------------------------------------------------------------- 40-layer slice

# Projections of one Llama-70B-shaped decoder layer (name, d_out, d_in): QKV
# 8192 -> 10240 (64 query and 8 key/value heads of 128), O 8192 -> 8192,
# gate+up 8192 -> 2 x 28672, down 28672 -> 8192.
SLICE_SHAPES = (("qkv", 10240, 8192), ("o", 8192, 8192), ("gate_up", 57344, 8192),
                ("down", 8192, 28672))
SLICE_SEED = 5
SLICE_PREFILL_TOKENS = 512
SLICE_DECODE_ROWS = 8


def slice_variant_scales(seed: int = SLICE_SEED):
    """Laplace scales of the slice's three fine-tuned variants (two resident,
    the third compressed layer by layer)."""
    from . import variant_scales
    return variant_scales(seed, 3)


def slice_base(layer: int, proj: int, seed: int = SLICE_SEED):
    """W_base of projection `proj` (index into SLICE_SHAPES) of layer `layer`."""
    _, d_out, d_in = SLICE_SHAPES[proj]
    return normal_bf16((d_out, d_in), seed, 10000 + 10 * layer + proj, SIGMA_BASE)


def slice_finetuned(wb: torch.Tensor, layer: int, proj: int, variant: int,
                    seed: int = SLICE_SEED, out: torch.Tensor = None):
    """W_ft of resident variant 1 or 2, or of variant 3 (the one compressed
    layer by layer), for one projection of the slice."""
    b = float(slice_variant_scales(seed)[variant - 1])
    if variant == 3:
        stream = 50000 + 10 * layer + proj
    else:
        stream = 20000 + 100 * layer + 10 * proj + (variant - 1)
    return finetuned_bf16(wb, seed, stream, b, out)


def slice_inputs(d_in: int, rows: int, decode: bool, seed: int = SLICE_SEED):
    """x of one projection's width: the 512-token prefill input or the 8-row
    decode batch (fresh N(0, 1) per width; projections are not chained)."""
    return normal_bf16((rows, d_in), seed, (40000 if decode else 30000) + d_in)
