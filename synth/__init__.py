"""Seeded synthetic inputs for the BitDelta hot path.

This module serves both the CUDA library's tests/benchmark and the CPU oracle.
It holds none of the method's arithmetic: it only draws random tensors and
converts them to bf16 bit patterns (through torch's own float32 -> bf16
conversion).  No delta, sign, alpha, reconstruction or product is computed
here.

Distributions follow the workloads the BitDelta page describes: base weights
W_base ~ N(0, 0.02) in bf16, fine-tuning deltas Δ ~ Laplace(0, b) (the page's
"Mathematical foundation" models Δ_ij as Laplace(0, b)), W_ft = bf16(W_base +
Δ), activations x ~ N(0, 1) in bf16.

Host generators (numpy PCG64, seeded) are used for sizes a host handles in
well under a second; ``synth.device`` draws the large workloads directly on the
GPU with a counter-based generator.
"""
from __future__ import annotations

import numpy as np
import torch

SIGMA_BASE = 0.02
LAPLACE_B = 1e-3


def bf16_bits(a) -> np.ndarray:
    """float32/float64 array -> bf16 bit patterns (uint16), via torch's RNE cast."""
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()


def bf16_to_f32(bits) -> np.ndarray:
    """bf16 bit patterns -> float32 values (exact widening)."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


def _rng(seed: int, stream: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64([int(seed), int(stream)]))


def base_weight(seed: int, d_out: int, d_in: int, sigma: float = SIGMA_BASE) -> np.ndarray:
    """W_base bf16 [d_out, d_in] ~ N(0, sigma)."""
    g = _rng(seed, 1)
    w = g.standard_normal((d_out, d_in), dtype=np.float32) * np.float32(sigma)
    return bf16_bits(w)


def finetuned_weight(seed: int, w_base: np.ndarray, b: float = LAPLACE_B,
                     stream: int = 2) -> np.ndarray:
    """W_ft = bf16(fp32(W_base + Δ)), Δ ~ Laplace(0, b) drawn in fp64."""
    g = _rng(seed, stream)
    delta = g.laplace(0.0, b, size=w_base.shape)
    ft = bf16_to_f32(w_base).astype(np.float64) + delta
    return bf16_bits(ft.astype(np.float32))


def layer(seed: int, d_out: int, d_in: int, sigma: float = SIGMA_BASE, b: float = LAPLACE_B):
    """(W_base, W_ft) bf16 bit patterns for one synthetic layer."""
    wb = base_weight(seed, d_out, d_in, sigma)
    return wb, finetuned_weight(seed, wb, b)


def activations(seed: int, M: int, d_in: int, stream: int = 3) -> np.ndarray:
    """x bf16 [M, d_in] ~ N(0, 1)."""
    g = _rng(seed, stream)
    return bf16_bits(g.standard_normal((M, d_in), dtype=np.float32))


def constant_magnitude_case(seed: int, d_out: int = 8, d_in: int = 16, log2_c: int = -10):
    """Inputs with |Δ_ij| == c exactly, c = 2**log2_c.

    W_base = k·c with integer k in [-127, 127] and W_ft = W_base ± c: every
    value has at most 8 significant bits, so all are exact in bf16 and the
    difference W_ft − W_base is exactly ±c.  Returns (W_base, W_ft, c).
    """
    g = _rng(seed, 4)
    c = 2.0 ** log2_c
    k = g.integers(-127, 128, size=(d_out, d_in)).astype(np.float64)
    s = np.where(g.integers(0, 2, size=(d_out, d_in)) == 1, 1.0, -1.0)
    wb = bf16_bits((k * c).astype(np.float32))
    wf = bf16_bits(((k + s) * c).astype(np.float32))
    return wb, wf, c


def segments(seed: int, lengths, n_var: int):
    """Row segments and variant ids for the multi-tenant linear.

    ``lengths`` lists the row count of each request; ids are drawn uniformly
    over {0 (base), 1..n_var}.  Returns (seg_offsets int32 [n_seg+1],
    seg_variant int32 [n_seg]).
    """
    g = _rng(seed, 5)
    lengths = np.asarray(lengths, dtype=np.int64)
    off = np.zeros(lengths.shape[0] + 1, np.int32)
    off[1:] = np.cumsum(lengths)
    var = g.integers(0, n_var + 1, size=lengths.shape[0]).astype(np.int32)
    return off, var


def variant_scales(seed: int, n_var: int, lo: float = 5e-4, hi: float = 2e-3) -> np.ndarray:
    """Per-variant Laplace scales b_v ~ U[lo, hi]."""
    g = _rng(seed, 6)
    return g.uniform(lo, hi, size=n_var)


def monosoup_checkpoints(seed: int, w_base: np.ndarray, k: int, rank: int,
                         s_hi: float = 1.0, s_lo: float = 0.5, noise_b: float = 1e-4):
    """k fine-tuned checkpoints W_i = bf16(W_base + Δ_i) for the MonoSoup merge.

    Following the page's MonoSoup section (fine-tuning moves a model along a
    few high-variance directions in weight space), each Δ_i is a rank-``rank``
    signal plus small dense noise: Σ_j s_j·a_j·b_jᵀ with s_j spaced
    geometrically from s_hi down to s_lo, a_j ~ N(0, 1/d_out) and
    b_j ~ N(0, 1/d_in) drawn independently (near-orthogonal, near-unit columns
    for d >> rank), plus Laplace(0, noise_b) per element.  Returns a list of
    bf16 bit-pattern arrays.
    """
    d_out, d_in = w_base.shape
    base = bf16_to_f32(w_base).astype(np.float64)
    s = np.geomspace(s_hi, s_lo, rank) if rank > 0 else np.zeros(0)
    out = []
    for i in range(k):
        g = _rng(seed, 100 + i)
        a = g.standard_normal((d_out, rank)) / np.sqrt(d_out)
        b = g.standard_normal((d_in, rank)) / np.sqrt(d_in)
        delta = (a * s) @ b.T + g.laplace(0.0, noise_b, size=(d_out, d_in))
        out.append(bf16_bits((base + delta).astype(np.float32)))
    return out
