"""Element-wise GPU parity of the decode kernels (M <= 16 and the short rows
of the grouped linear) with deltas as large as the weights.

The decode kernels compute the exact split y = x·W_baseᵀ + α ⊙ (x·Sᵀ) (the
effective weight W_base + α·sign(Δ) of the page's "Mathematical foundation",
not rounded to bf16), so they are compared with the oracle's split form,
element by element, under

    |y − y_ref| <= 2^-8·|y_ref| + (d_in/16 + 8)·2^-21·(Σ_k|x_k·W_base,k| + α·Σ_k|x_k|)

(bf16 rounding of the output, half an ulp; fp32 accumulation over d_in/16
tensor-core steps, each allowed eight fp32 roundings of the running sums,
plus the cross-warp sum and the α multiply-add).  With Δ ~ Laplace(0, 0.02)
the sign term is as large as the base term, so a sign product dropped or
misplaced over any 32-column chunk (about α·√32 ≈ 0.1) fails the bound
(about 0.015 at d_in = 1024), where the 1e-2·max|y_ref| bar would not notice
it.  The rows also meet that bar against the rounded oracle linear.
"""
import numpy as np
import pytest

import bit_weight_delta_gb300 as bd
import oracle
import synth
from gpu_util import assert_linear_close, bf16_values, to_dev, to_dev_bf16

pytestmark = pytest.mark.gpu

BIG_B = 0.02


def _bound(x, wb, alpha_rows, d_in):
    xa = np.abs(synth.bf16_to_f32(x).astype(np.float64))
    A = xa @ np.abs(synth.bf16_to_f32(wb).astype(np.float64)).T
    B = xa.sum(axis=1, keepdims=True)
    return (d_in / 16 + 8) * 2.0 ** -21 * (A + B * alpha_rows[None, :])


def _assert_elementwise(y, ref, acc_bound, what):
    bound = 2.0 ** -8 * np.abs(ref) + acc_bound
    err = np.abs(y - ref)
    bad = err > bound
    assert not bad.any(), (f"{what}: {int(bad.sum())} of {bad.size} outputs off, worst "
                           f"{float((err - bound).max()):.3e} over the bound")


def _layer(seed, d_out, d_in, per_row):
    wb = synth.base_weight(seed, d_out, d_in)
    wf = synth.finetuned_weight(seed, wb, b=BIG_B, stream=7)
    packed, alpha = oracle.compress(wb, wf, per_row)[:2]
    return wb, packed, alpha


@pytest.mark.parametrize("per_row", [True, False])
@pytest.mark.parametrize("M", [1, 3, 8, 9, 16])
@pytest.mark.parametrize("d_in,d_out", [(1024, 600), (1032, 600), (1024, 5000)])
def test_decode_linear_elementwise(M, d_in, d_out, per_row):
    """d_in = 1024: 16-byte sign rows (the cp.async ring for M <= 8, and for
    9..16 on the one-wave grid of d_out = 600; d_out = 5000 is a grid of more
    than two CTAs per SM, where 9..16 take the register pipeline); d_in =
    1032: sign rows not 16-byte aligned (byte-wise sign loads, a 32-column
    tail).  d_out = 600 and 5000: a partial last group of 16 rows."""
    wb, packed, alpha = _layer(31 + M, d_out, d_in, per_row)
    x = synth.activations(31 + M, M, d_in)
    y = bf16_values(bd.bitdelta_linear(to_dev_bf16(x), to_dev_bf16(wb), to_dev(packed),
                                       to_dev(alpha), per_row=per_row))
    assert bd.bitdelta_check_error() == 0
    ref = oracle.linear_split(x, wb, packed, alpha, per_row)
    a_rows = alpha.astype(np.float64) if per_row else np.full(d_out, float(alpha[0]))
    _assert_elementwise(y, ref, _bound(x, wb, a_rows, d_in), f"M={M} d_in={d_in}")
    assert_linear_close(y, oracle.linear(x, wb, packed, alpha, per_row), f"M={M}")


@pytest.mark.parametrize("d_in", [1024, 520])
def test_grouped_short_rows_elementwise(d_in):
    """Short segments only (every row on the decode kernel), five variants
    plus base rows, more than 16 rows in all so several groups form; each
    output compared with the split form of its own variant."""
    d_out, n_var = 300, 5
    wb = synth.base_weight(41, d_out, d_in)
    packs, alphas = [], []
    for v in range(n_var):
        wf = synth.finetuned_weight(41, wb, b=BIG_B * (0.5 + 0.25 * v), stream=200 + v)
        p, a = oracle.compress(wb, wf, True)[:2]
        packs.append(p)
        alphas.append(a)
    lengths = [1, 3, 1, 5, 2, 1, 4, 1, 2, 3, 1, 1]
    var = np.array([1, 0, 2, 3, 5, 1, 4, 0, 2, 5, 3, 4], np.int32)
    off = np.zeros(len(lengths) + 1, np.int32)
    off[1:] = np.cumsum(lengths)
    x = synth.activations(41, int(off[-1]), d_in)
    dp, da = [to_dev(p) for p in packs], [to_dev(a) for a in alphas]   # alive while used
    pt, at = bd.variant_tables(dp, da, "cuda")
    y = bf16_values(bd.bitdelta_linear_grouped(
        to_dev_bf16(x), to_dev(off), to_dev(var), to_dev_bf16(wb), pt, at, n_var=n_var,
        max_seg_len=int(np.diff(off).max()), per_row=True))
    assert bd.bitdelta_check_error() == 0
    zero = np.zeros(d_out, np.float32)
    for s in range(len(lengths)):
        rows = slice(off[s], off[s + 1])
        v = int(var[s])
        p = packs[v - 1] if v else packs[0]
        a = alphas[v - 1] if v else zero
        ref = oracle.linear_split(x[rows], wb, p, a, True)
        _assert_elementwise(y[rows], ref, _bound(x[rows], wb, a.astype(np.float64), d_in),
                            f"segment {s} (variant {v})")
    assert_linear_close(y, oracle.linear_grouped(x, off, var, wb, packs, alphas, True))


@pytest.mark.parametrize("d_out,d_in,per_row,shift", [(5000, 16384, True, 0),
                                                     (8192, 16512, False, 0),
                                                     (5000, 16384, True, 8),
                                                     (4864, 16384, True, 0),
                                                     (5000, 1024, True, 0)])
def test_grouped_two_variants_pair_split_elementwise(d_out, d_in, per_row, shift):
    """Eight one-row segments alternating two variants (the 40-layer slice's
    decode batch) on layers of 313 and 512 row blocks with d_in >= 16384,
    whose grids the host splits over d_in between the two CTAs of a cluster
    (CTA 1's sums added to CTA 0's through distributed shared memory; 16512
    leaves the two CTAs unequal runs of stages), and without the split (304
    blocks; d_in = 1024): every output against the split form of its own
    variant.  shift = 8: variant 2's sign table starts 8 bytes past a 16-byte
    boundary (its words fetched with plain loads)."""
    import torch
    n_var = 2
    wb = synth.base_weight(42, d_out, d_in)
    packs, alphas = [], []
    for v in range(n_var):
        wf = synth.finetuned_weight(42, wb, b=BIG_B * (0.6 + 0.4 * v), stream=300 + v)
        p, a = oracle.compress(wb, wf, per_row)[:2]
        packs.append(p)
        alphas.append(a)
    off = np.arange(9, dtype=np.int32)
    var = np.array([1 + (r % 2) for r in range(8)], np.int32)
    x = synth.activations(42, 8, d_in)
    dp, da = [to_dev(p) for p in packs], [to_dev(a) for a in alphas]
    keep = []
    if shift:
        raw = torch.empty(packs[1].size + 16, dtype=torch.uint8, device="cuda")
        shifted = raw[shift:shift + packs[1].size].view(packs[1].shape)
        shifted.copy_(dp[1])
        assert shifted.data_ptr() % 16 == shift
        keep.append(raw)
        dp[1] = shifted
    pt, at = bd.variant_tables(dp, da, "cuda")
    y = bf16_values(bd.bitdelta_linear_grouped(
        to_dev_bf16(x), to_dev(off), to_dev(var), to_dev_bf16(wb), pt, at, n_var=n_var,
        max_seg_len=1, per_row=per_row))
    assert bd.bitdelta_check_error() == 0
    for r in range(8):
        v = int(var[r])
        a = alphas[v - 1]
        a_rows = (a if per_row else np.full(d_out, a[0], np.float32)).astype(np.float64)
        ref = oracle.linear_split(x[r:r + 1], wb, packs[v - 1], a, per_row)
        _assert_elementwise(y[r:r + 1], ref, _bound(x[r:r + 1], wb, a_rows, d_in),
                            f"row {r} (variant {v})")
