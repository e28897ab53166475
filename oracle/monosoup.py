"""MonoSoup merge, plain fp64 oracle (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` use this module.  It shares no code with the CUDA library.

Page "BitDelta: serving 14 Zen models from one GPU cluster", section
"MonoSoup: complementing the single checkpoint with SVD": given k fine-tuned
checkpoints W_1..W_k of one base W_base,
    Δ_i = W_i − W_base,
    τ_i = the rank-r truncated SVD of Δ_i, U_i[:, :r] · diag(S_i[:r]) · Vh_i[:r],
    W_merged = W_base + (1/k) · Σ_i τ_i.
The truncation is read as the exact one (the best rank-r approximation of
Δ_i in the Frobenius norm).  The SVD itself is LAPACK's, through
``numpy.linalg.svd``, used as a library step; everything else is written out
below in fp64.  W_merged is stored as bf16, rounded once from the fp64 value
to the nearest bf16 (ties to even).

All bf16 tensors are numpy ``uint16`` bit patterns.
"""
from __future__ import annotations

import numpy as np


def bf16_to_f64(bits) -> np.ndarray:
    """bf16 bit patterns -> float64 values (exact)."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def bf16_rne(x) -> np.ndarray:
    """float64 values -> bf16 bit patterns, rounded to nearest, ties to even.

    bf16 keeps 8 significant bits and the float32 exponent range: a normal
    value x = m·2^e (0.5 <= |m| < 1) rounds to rint(m·2^8)·2^(e-8); below the
    normal range the spacing stays 2^-133.  numpy's rint rounds halves to
    even.  Finite inputs only.
    """
    x = np.asarray(x, dtype=np.float64)
    _, e = np.frexp(x)
    e = np.maximum(e, -125)
    y = np.ldexp(np.rint(np.ldexp(x, 8 - e)), e - 8)
    return (y.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)


def truncated_svd(delta: np.ndarray, rank: int) -> np.ndarray:
    """τ = U[:, :r] · diag(S[:r]) · Vh[:r] of delta (fp64)."""
    delta = np.asarray(delta, dtype=np.float64)
    if rank <= 0:
        return np.zeros_like(delta)
    u, s, vh = np.linalg.svd(delta, full_matrices=False)
    r = min(rank, s.shape[0])
    return (u[:, :r] * s[:r]) @ vh[:r]


def monosoup(w_base_bits, w_ft_bits_list, rank: int):
    """MonoSoup merge of the checkpoints in ``w_ft_bits_list`` over ``w_base_bits``.

    Returns (W_merged bf16 bits, W_merged fp64 before rounding,
    correction fp64 = (1/k)·Σ τ_i).
    """
    k = len(w_ft_bits_list)
    if k < 1:
        raise ValueError("MonoSoup needs at least one checkpoint")
    wb = bf16_to_f64(w_base_bits)
    correction = np.zeros_like(wb)
    for w in w_ft_bits_list:
        delta = bf16_to_f64(w) - wb          # exact: both are bf16 values
        correction += truncated_svd(delta, rank)
    correction /= k
    merged = wb + correction
    return bf16_rne(merged), merged, correction
