"""GPU parity of the wide short-row pass of bitdelta_linear_grouped (more short
rows than one 16-row group: up to 64 rows of up to 16 delta variants per pass
over W_base), element by element against the oracle's split form
("Serving architecture": base weights shared-read by every variant, the
request's model id selects the delta; the effective weight of "Mathematical
foundation").

Deltas are as large as the weights (Laplace(0, 0.02)), so a sign product
credited to the wrong token, variant, tile or chunk, or an α taken from the
wrong row, misses the element-wise bound by far.  Cases: several passes, a
pass closed early at the variant cap, one variant spanning several tiles,
base rows between variants, a partial last block of output rows, per-matrix
α, sign tables off a 16-byte boundary, and short rows next to long segments
(few short rows with a large host bound included).
"""
import numpy as np
import pytest
import torch

import bit_weight_delta_gb300 as bd
import oracle
import synth
from gpu_util import (assert_linear_close, assert_split_elementwise, bf16_values, to_dev,
                      to_dev_bf16)

pytestmark = pytest.mark.gpu

BIG_B = 0.02


def _variants(seed, wb, n_var, per_row):
    packs, alphas = [], []
    for v in range(n_var):
        wf = synth.finetuned_weight(seed, wb, b=BIG_B * (0.5 + 0.05 * v), stream=400 + v)
        p, a = oracle.compress(wb, wf, per_row)[:2]
        packs.append(p)
        alphas.append(a)
    return packs, alphas


def _offsets(lengths):
    off = np.zeros(len(lengths) + 1, np.int32)
    off[1:] = np.cumsum(lengths)
    return off


def _call(x, off, var, wb, dp, da, n_var, per_row):
    pt, at = bd.variant_tables(dp, da, "cuda")
    y = bd.bitdelta_linear_grouped(to_dev_bf16(x), to_dev(off), to_dev(var), to_dev_bf16(wb), pt,
                                   at, n_var=n_var, max_seg_len=int(np.diff(off).max()),
                                   per_row=per_row)
    assert bd.bitdelta_check_error() == 0
    return bf16_values(y)


def _check_segments(y, x, off, var, wb, packs, alphas, per_row, short_max=16):
    d_out = wb.shape[0]
    zero = np.zeros(d_out if per_row else 1, np.float32)
    for s in range(len(var)):
        rows = slice(int(off[s]), int(off[s + 1]))
        if off[s + 1] == off[s]:
            continue
        v = int(var[s])
        p = packs[v - 1] if v else packs[0]
        a = alphas[v - 1] if v else zero
        if off[s + 1] - off[s] <= short_max:
            assert_split_elementwise(y[rows], x[rows], wb, p, a, per_row,
                                     f"segment {s} (variant {v})")
        else:  # long segments: the tensor-core kernel's rounded W_eff
            assert_linear_close(y[rows], oracle.linear(x[rows], wb, p, a, per_row),
                                f"segment {s} (variant {v})")


@pytest.mark.parametrize("per_row", [True, False])
def test_wide_many_rows_many_variants(per_row):
    """150 one-row segments over 20 variants and base: passes of at most 64
    rows, some closed early because a 17th variant would join; d_out = 600
    leaves a partial last block of 16 output rows."""
    d_out, d_in, n_var = 600, 1024, 20
    wb = synth.base_weight(71, d_out, d_in)
    packs, alphas = _variants(71, wb, n_var, per_row)
    rng = np.random.default_rng(71)
    lengths = [1] * 150
    var = rng.integers(0, n_var + 1, size=len(lengths)).astype(np.int32)
    off = _offsets(lengths)
    x = synth.activations(71, int(off[-1]), d_in)
    dp, da = [to_dev(p) for p in packs], [to_dev(a) for a in alphas]
    y = _call(x, off, var, wb, dp, da, n_var, per_row)
    _check_segments(y, x, off, var, wb, packs, alphas, per_row)


def test_wide_one_variant_across_tiles_with_base_rows():
    """Short segments of up to 16 rows: variant 2 holds 29 rows (four tiles),
    variant 5 a single row, base rows on both sides."""
    d_out, d_in, n_var = 256, 512, 5
    wb = synth.base_weight(72, d_out, d_in)
    packs, alphas = _variants(72, wb, n_var, True)
    lengths = [3, 16, 13, 1, 4, 2, 7]
    var = np.array([0, 2, 2, 5, 0, 1, 3], np.int32)
    off = _offsets(lengths)
    x = synth.activations(72, int(off[-1]), d_in)
    dp, da = [to_dev(p) for p in packs], [to_dev(a) for a in alphas]
    y = _call(x, off, var, wb, dp, da, n_var, True)
    _check_segments(y, x, off, var, wb, packs, alphas, True)


@pytest.mark.parametrize("shift", [1, 8])
def test_wide_unaligned_sign_tables(shift):
    """Two of six variants have packed signs starting `shift` bytes past a
    16-byte boundary (fetched with plain loads), the others by cp.async."""
    d_out, d_in, n_var = 320, 1024, 6
    wb = synth.base_weight(73, d_out, d_in)
    packs, alphas = _variants(73, wb, n_var, True)
    dp = [to_dev(p) for p in packs]
    keep = []
    for v in (1, 4):
        raw = torch.empty(packs[v].size + 16, dtype=torch.uint8, device="cuda")
        shifted = raw[shift:shift + packs[v].size].view(packs[v].shape)
        shifted.copy_(dp[v])
        assert shifted.data_ptr() % 16 == shift
        keep.append(raw)
        dp[v] = shifted
    da = [to_dev(a) for a in alphas]
    lengths = [1] * 40
    var = (np.arange(40) % (n_var + 1)).astype(np.int32)
    off = _offsets(lengths)
    x = synth.activations(73, int(off[-1]), d_in)
    y = _call(x, off, var, wb, dp, da, n_var, True)
    _check_segments(y, x, off, var, wb, packs, alphas, True)


@pytest.mark.parametrize("n_short", [3, 70])
def test_wide_short_rows_beside_long_segments(n_short):
    """Long segments on the tensor-core kernel and short rows on the wide
    pass; with 3 short rows the host's bound (16 per segment) still selects
    the wide pass, which then runs one token tile."""
    d_out, d_in, n_var = 384, 1024, 7
    wb = synth.base_weight(74, d_out, d_in)
    packs, alphas = _variants(74, wb, n_var, False)
    rng = np.random.default_rng(74 + n_short)
    lengths = [300, 1, 200] + [1] * (n_short - 1) + [257]
    var = rng.integers(0, n_var + 1, size=len(lengths)).astype(np.int32)
    off = _offsets(lengths)
    x = synth.activations(74, int(off[-1]), d_in)
    dp, da = [to_dev(p) for p in packs], [to_dev(a) for a in alphas]
    y = _call(x, off, var, wb, dp, da, n_var, False)
    _check_segments(y, x, off, var, wb, packs, alphas, False)


@pytest.mark.parametrize("shape,n_var,n_rows,per_row", [
    ((12500, 256), 10, 150, True),   # 782 blocks of 16 rows, the last one of 4 rows
    ((10000, 384), 20, 70, False),   # 625 blocks
])
def test_wide_pass_multi_wave_layers(shape, n_var, n_rows, per_row):
    """Layers of several CTA waves (more than four 16-row blocks per SM):
    a partial last block, several passes and the variant cap, element-wise."""
    d_out, d_in = shape
    wb = synth.base_weight(75, d_out, d_in)
    packs, alphas = _variants(75, wb, n_var, per_row)
    rng = np.random.default_rng(75 + d_out)
    var = rng.integers(0, n_var + 1, size=n_rows).astype(np.int32)
    off = _offsets([1] * n_rows)
    x = synth.activations(75, int(off[-1]), d_in)
    dp, da = [to_dev(p) for p in packs], [to_dev(a) for a in alphas]
    y = _call(x, off, var, wb, dp, da, n_var, per_row)
    _check_segments(y, x, off, var, wb, packs, alphas, per_row)


def test_wide_pass_multi_wave_unaligned_signs_and_segments():
    """A multi-wave layer with one variant's signs 8 bytes off a 16-byte boundary,
    short segments of several rows (one variant over several tiles) and a
    long segment on the tensor-core kernel."""
    d_out, d_in, n_var = 12500, 256, 4
    wb = synth.base_weight(76, d_out, d_in)
    packs, alphas = _variants(76, wb, n_var, True)
    dp = [to_dev(p) for p in packs]
    raw = torch.empty(packs[2].size + 16, dtype=torch.uint8, device="cuda")
    shifted = raw[8:8 + packs[2].size].view(packs[2].shape)
    shifted.copy_(dp[2])
    dp[2] = shifted
    da = [to_dev(a) for a in alphas]
    lengths = [16, 9, 1, 300, 12, 16, 3]
    var = np.array([3, 3, 0, 1, 2, 4, 3], np.int32)
    off = _offsets(lengths)
    x = synth.activations(76, int(off[-1]), d_in)
    y = _call(x, off, var, wb, dp, da, n_var, True)
    _check_segments(y, x, off, var, wb, packs, alphas, True)
