"""GPU parity: bitdelta_compress and bitdelta_reconstruct against the oracle.

Signs, packing and the reconstructed bf16 weight must be bit-exact; α within
1e-6 relative of the oracle's fp64 mean|Δ| ("Mathematical foundation")."""
import numpy as np
import pytest
import torch

import bit_weight_delta_gb300 as bd
import oracle
import synth
from gpu_util import ALPHA_RTOL, from_dev_bf16, to_dev_bf16

pytestmark = pytest.mark.gpu

# (d_out, d_in): the tiny config, the decode layer, ragged rows and columns
SHAPES = [(256, 512), (4096, 4096), (8, 16), (1, 8), (3, 24), (37, 136), (130, 1032), (513, 256)]


def _check_compress(wb, wf, per_row):
    packed_ref, a32_ref, a64_ref = oracle.compress(wb, wf, per_row)
    packed, alpha = bd.bitdelta_compress(to_dev_bf16(wb), to_dev_bf16(wf), per_row=per_row)
    assert bd.bitdelta_check_error() == 0
    assert np.array_equal(packed.cpu().numpy(), packed_ref)
    a = alpha.cpu().numpy().astype(np.float64)
    rel = np.abs(a - a64_ref) / np.maximum(np.abs(a64_ref), 1e-300)
    assert (rel <= ALPHA_RTOL).all(), rel.max()
    return packed, alpha


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("per_row", [True, False])
def test_compress_matches_oracle(shape, per_row):
    d_out, d_in = shape
    wb, wf = synth.layer(0, d_out, d_in)
    _check_compress(wb, wf, per_row)


def test_compress_constant_magnitude_exact():
    """|Δ| ≡ c: α == c exactly and reconstruct returns W_ft bit for bit."""
    for seed in range(3):
        wb, wf, c = synth.constant_magnitude_case(seed, 8, 16)
        for per_row in (True, False):
            packed, alpha = bd.bitdelta_compress(to_dev_bf16(wb), to_dev_bf16(wf), per_row=per_row)
            assert (alpha.cpu().numpy() == np.float32(c)).all()
            w = bd.bitdelta_reconstruct(to_dev_bf16(wb), packed, alpha, per_row=per_row)
            assert np.array_equal(from_dev_bf16(w), wf)


def test_compress_zero_delta_and_signed_zeros():
    wb = np.full((4, 64), 0x3E00, np.uint16)   # 0.125
    wb[0, :8] = 0x8000                         # −0 base
    wf = wb.copy()
    wf[0, :8] = 0x0000                         # +0 fine-tuned: Δ = +0 - (−0) = 0 -> +1
    wf[1, 8:16] = 0x8000                       # W_ft −0 against 0.125: negative
    _check_compress(wb, wf, True)
    _check_compress(wb, wf, False)


def test_compress_deterministic():
    wb, wf = synth.layer(9, 1024, 2048)
    a = [bd.bitdelta_compress(to_dev_bf16(wb), to_dev_bf16(wf), per_row=False)[1].item()
         for _ in range(3)]
    assert a[0] == a[1] == a[2]


def test_compress_workspace_reuse():
    """Two per-matrix calls in a row through one caller workspace."""
    wb, wf = synth.layer(4, 300, 512)
    ws = torch.empty(bd.bitdelta_compress_workspace_bytes(300, 512, False), dtype=torch.uint8,
                     device="cuda")
    _, ref, _ = oracle.compress(wb, wf, False)
    for _ in range(2):
        _, alpha = bd.bitdelta_compress(to_dev_bf16(wb), to_dev_bf16(wf), per_row=False,
                                        workspace=ws)
        assert abs(alpha.item() - ref[0]) <= ALPHA_RTOL * ref[0]


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("per_row", [True, False])
def test_reconstruct_bit_exact(shape, per_row):
    """The oracle is fed the GPU's α so both sides add the same fp32 value."""
    d_out, d_in = shape
    wb, wf = synth.layer(1, d_out, d_in)
    packed, alpha = bd.bitdelta_compress(to_dev_bf16(wb), to_dev_bf16(wf), per_row=per_row)
    w = bd.bitdelta_reconstruct(to_dev_bf16(wb), packed, alpha, per_row=per_row)
    assert bd.bitdelta_check_error() == 0
    ref = oracle.reconstruct(wb, packed.cpu().numpy(), alpha.cpu().numpy(), per_row)
    assert np.array_equal(from_dev_bf16(w), ref)


def test_reconstruct_alpha_zero_and_negative_zero():
    wb, wf = synth.layer(2, 16, 64)
    wb = wb.copy()
    wb[0, :16] = 0x8000
    packed, _ = bd.bitdelta_compress(to_dev_bf16(wb), to_dev_bf16(wf), per_row=True)
    alpha = torch.zeros(16, dtype=torch.float32, device="cuda")
    w = bd.bitdelta_reconstruct(to_dev_bf16(wb), packed, alpha, per_row=True)
    ref = oracle.reconstruct(wb, packed.cpu().numpy(), alpha.cpu().numpy(), True)
    assert np.array_equal(from_dev_bf16(w), ref)
