"""Helpers for the GPU parity tests: host bf16 bit arrays <-> CUDA tensors, and
the linear-output tolerance max|y − y_ref| <= 1e-2 · max|y_ref|."""
import numpy as np
import torch

import synth

LINEAR_RTOL = 1e-2     # max|y − y_ref| <= LINEAR_RTOL · max|y_ref| (fp32 accumulation)
ALPHA_RTOL = 1e-6      # α relative to the fp64 oracle


def to_dev_bf16(bits: np.ndarray) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(bits, dtype=np.uint16).view(np.int16))
    return t.view(torch.bfloat16).cuda()


def from_dev_bf16(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def bf16_values(t: torch.Tensor) -> np.ndarray:
    return synth.bf16_to_f32(from_dev_bf16(t)).astype(np.float64)


def to_dev(a: np.ndarray, dtype=None) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.to(dtype)
    return t.cuda()


def assert_linear_close(y_gpu: np.ndarray, y_ref: np.ndarray, what: str = ""):
    y_gpu = np.asarray(y_gpu, dtype=np.float64)
    y_ref = np.asarray(y_ref, dtype=np.float64)
    assert y_gpu.shape == y_ref.shape, (y_gpu.shape, y_ref.shape)
    assert np.isfinite(y_gpu).all(), f"{what}: non-finite output"
    scale = np.abs(y_ref).max()
    err = np.abs(y_gpu - y_ref).max()
    assert err <= LINEAR_RTOL * scale, f"{what}: max err {err:.3e} > {LINEAR_RTOL} * {scale:.3e}"
    return err / scale if scale > 0 else err


def assert_split_elementwise(y, x, wb, packed, alpha, per_row: bool, what: str = ""):
    """Element-wise bound for the kernels that compute the exact split
    y = x·W_baseᵀ + α ⊙ (x·Sᵀ) (W_eff not rounded to bf16): against the
    oracle's split form,
        |y − y_ref| <= 2^-8·|y_ref| + (d_in/16 + 8)·2^-21·(Σ_k|x_k·W_base,k| + α·Σ_k|x_k|)
    (bf16 rounding of the output, half an ulp, and fp32 accumulation over
    d_in/16 tensor-core steps, each allowed eight roundings of the running
    sums)."""
    import oracle
    d_out, d_in = wb.shape
    y = np.asarray(y, dtype=np.float64)
    ref = oracle.linear_split(x, wb, packed, alpha, per_row)
    xa = np.abs(synth.bf16_to_f32(x).astype(np.float64))
    a_rows = alpha.astype(np.float64) if per_row else np.full(d_out, float(alpha[0]))
    acc = (d_in / 16 + 8) * 2.0 ** -21 * (
        xa @ np.abs(synth.bf16_to_f32(wb).astype(np.float64)).T
        + xa.sum(axis=1, keepdims=True) * a_rows[None, :])
    err = np.abs(y - ref)
    bound = 2.0 ** -8 * np.abs(ref) + acc
    bad = err > bound
    assert not bad.any(), (f"{what}: {int(bad.sum())} of {bad.size} outputs off, worst "
                           f"{float((err - bound).max()):.3e} over the bound")
