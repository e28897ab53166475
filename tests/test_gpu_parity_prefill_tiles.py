"""GPU parity of the prefill kernel's two tile widths (256 and 512 tokens per
CTA-pair tile) against the oracle, with deltas as large as the weights.

Page section "Serving architecture": y = x·(W_base + α·unpack(bits))ᵀ with
W_eff built on chip.  The 512-token tile writes W_eff back over W_base in
shared memory; a stage whose MMA saw W_base instead would change y by
α·Σ±x over that stage's 64 columns.  With Δ ~ Laplace(0, 0.02) (α about the
size of |W_base|) that is ~0.16 against the element-wise bound used here:

    |y − y_ref| <= 2^-8·|y_ref| + d_in·2^-22·Σ_k |x_k|·|W_eff,k|

(bf16 rounding of the output, half an ulp at most 2^-8 relative, plus a
generous bound on the fp32 accumulation of exact bf16 products), so one
stale stage anywhere fails the test, while the 1e-2·max|y_ref| bar alone
would not notice it.
"""
import numpy as np
import pytest

import bit_weight_delta_gb300 as bd
import oracle
import synth
from gpu_util import assert_linear_close, bf16_values, to_dev, to_dev_bf16

pytestmark = pytest.mark.gpu

BIG_B = 0.02   # Laplace scale of Δ, equal to the base weights' σ


def _weff(wb, packed, alpha, per_row):
    return synth.bf16_to_f32(oracle.reconstruct(wb, packed, alpha, per_row)).astype(np.float64)


def _assert_elementwise(y, ref, absmag, d_in, what=""):
    bound = 2.0 ** -8 * np.abs(ref) + d_in * 2.0 ** -22 * absmag
    err = np.abs(y - ref)
    bad = err > bound
    assert not bad.any(), (f"{what}: {int(bad.sum())} outputs off, worst "
                           f"{float((err - bound).max()):.3e} over the bound")


def _big_layer(seed, d_out, d_in, per_row, stream=2):
    wb = synth.base_weight(seed, d_out, d_in)
    wf = synth.finetuned_weight(seed, wb, b=BIG_B, stream=stream)
    packed, alpha = oracle.compress(wb, wf, per_row)[:2]
    return wb, packed, alpha


def _linear(x, wb, packed, alpha, per_row):
    return bf16_values(bd.bitdelta_linear(to_dev_bf16(x), to_dev_bf16(wb), to_dev(packed),
                                          to_dev(alpha), per_row=per_row))


@pytest.fixture(params=[256, 512])
def tile(request):
    """Each test runs with both pair-tile widths forced."""
    bd.bitdelta_set_prefill_tile(request.param)
    yield request.param
    bd.bitdelta_set_prefill_tile("auto")


@pytest.mark.parametrize("per_row", [True, False])
@pytest.mark.parametrize("M", [1100, 1023])
def test_tiles_elementwise(M, per_row, tile):
    """M = 1100 in 512-token tiles leaves a last tile of 76 tokens (its
    second MMA is skipped), M = 1023 one of 511.  d_out = 600 leaves a
    partial pair tile whose second CTA lies wholly past d_out."""
    d_out, d_in = 600, 1024
    wb, packed, alpha = _big_layer(21, d_out, d_in, per_row)
    x = synth.activations(21, M, d_in)
    y = _linear(x, wb, packed, alpha, per_row)
    assert bd.bitdelta_check_error() == 0
    ref = oracle.linear(x, wb, packed, alpha, per_row)
    assert_linear_close(y, ref, f"M={M}")
    xa = np.abs(synth.bf16_to_f32(x).astype(np.float64))
    absmag = xa @ np.abs(_weff(wb, packed, alpha, per_row)).T
    _assert_elementwise(y, ref, absmag, d_in, f"M={M}")


@pytest.mark.parametrize("d_in", [384, 640])
def test_tiles_persistent_loop(d_in, tile):
    """40 row tiles x 3 (or 5) token tiles: more tiles than the pairs of one
    GPU, so pairs take two or more; K-block counts that are not multiples of
    the ring's stages or of the two transform warpgroups (a warpgroup's
    stages cross tile boundaries)."""
    d_out, M = 256 * 40, 1030
    wb, packed, alpha = _big_layer(22, d_out, d_in, True)
    x = synth.activations(22, M, d_in)
    y = _linear(x, wb, packed, alpha, True)
    assert bd.bitdelta_check_error() == 0
    rng = np.random.default_rng(d_in)
    mi = rng.integers(0, M, 4000)
    ni = rng.integers(0, d_out, 4000)
    ref = oracle.linear_at(x, wb, packed, alpha, True, mi, ni)
    weff = _weff(wb, packed, alpha, True)
    xa = np.abs(synth.bf16_to_f32(x).astype(np.float64))
    absmag = np.einsum("ik,ik->i", xa[mi], np.abs(weff[ni]))
    _assert_elementwise(y[mi, ni], ref, absmag, d_in, f"d_in={d_in}")
    for m in (0, 511, 512, 1023, 1024, 1029):   # whole rows at tile edges
        ref_m = oracle.linear(x[m:m + 1], wb, packed, alpha, True)[0]
        _assert_elementwise(y[m], ref_m, xa[m] @ np.abs(weff).T, d_in, f"row {m}")


def test_tiles_grouped_segments(tile):
    """Grouped batch: a long delta segment ending mid-tile, a long base
    segment (no transform: the W_base stage is the operand as loaded), a
    600-token segment, and short rows between them on the decode kernel."""
    d_out, d_in, n_var = 300, 512, 3
    wb = synth.base_weight(23, d_out, d_in)
    packs, alphas, weffs = [], [], [synth.bf16_to_f32(wb).astype(np.float64)]
    for v in range(n_var):
        wf = synth.finetuned_weight(23, wb, b=BIG_B, stream=100 + v)
        p, a = oracle.compress(wb, wf, True)[:2]
        packs.append(p)
        alphas.append(a)
        weffs.append(_weff(wb, p, a, True))
    lengths = [1100, 3, 1, 1500, 600, 2]
    var = np.array([1, 2, 0, 0, 3, 1], np.int32)
    off = np.zeros(len(lengths) + 1, np.int32)
    off[1:] = np.cumsum(lengths)
    x = synth.activations(23, int(off[-1]), d_in)
    dp = [to_dev(p) for p in packs]
    da = [to_dev(a) for a in alphas]
    pt, at = bd.variant_tables(dp, da, "cuda")
    y = bf16_values(bd.bitdelta_linear_grouped(
        to_dev_bf16(x), to_dev(off), to_dev(var), to_dev_bf16(wb), pt, at, n_var=n_var,
        max_seg_len=int(np.diff(off).max()), per_row=True))
    assert bd.bitdelta_check_error() == 0
    ref = oracle.linear_grouped(x, off, var, wb, packs, alphas, True)
    assert_linear_close(y, ref)
    xa = np.abs(synth.bf16_to_f32(x).astype(np.float64))
    for s in range(len(lengths)):
        rows = slice(off[s], off[s + 1])
        if lengths[s] <= 16:
            # short rows run the decode kernel's exact split
            # x·W_baseᵀ + α·(x·Sᵀ), which does not round W_eff to bf16: the
            # 1e-2·max|y_ref| bar above is theirs
            continue
        absmag = xa[rows] @ np.abs(weffs[var[s]]).T
        _assert_elementwise(y[rows], ref[rows], absmag, d_in, f"segment {s}")


def test_tile_widths_agree():
    """Both widths accumulate the same K steps in the same order into fp32,
    one RNE rounding at the end: their outputs are expected to be identical
    bit for bit (checked here, on a problem of several tiles of each)."""
    d_out, d_in, M = 1000, 768, 1500
    wb, packed, alpha = _big_layer(24, d_out, d_in, True)
    x = synth.activations(24, M, d_in)
    out = {}
    try:
        for t in (256, 512):
            bd.bitdelta_set_prefill_tile(t)
            out[t] = _linear(x, wb, packed, alpha, True)
    finally:
        bd.bitdelta_set_prefill_tile("auto")
    assert bd.bitdelta_check_error() == 0
    diff = out[256] != out[512]
    assert not diff.any(), f"{int(diff.sum())} of {diff.size} outputs differ between widths"


@pytest.mark.parametrize("M", [2048, 2000])
def test_small_last_round_on_narrow_tiles(M):
    """40 row tiles x 4 token tiles of 512: on 76 CTA pairs two full rounds of
    512-token tiles, and the last round's 8 tiles (row tiles 38-39) run as 16
    tiles of 256 tokens in a second launch; M = 2000 leaves the last token
    tile of each row ragged.  Sampled outputs everywhere plus whole token rows,
    which cross both launches' row tiles, element-wise."""
    d_out, d_in = 256 * 40, 256
    wb, packed, alpha = _big_layer(25, d_out, d_in, True)
    x = synth.activations(25, M, d_in)
    y = _linear(x, wb, packed, alpha, True)
    assert bd.bitdelta_check_error() == 0
    weff = _weff(wb, packed, alpha, True)
    xa = np.abs(synth.bf16_to_f32(x).astype(np.float64))
    rng = np.random.default_rng(M)
    mi = rng.integers(0, M, 4000)
    ni = np.concatenate([rng.integers(0, d_out, 3000), rng.integers(38 * 256, d_out, 1000)])
    ref = oracle.linear_at(x, wb, packed, alpha, True, mi, ni)
    absmag = np.einsum("ik,ik->i", xa[mi], np.abs(weff[ni]))
    _assert_elementwise(y[mi, ni], ref, absmag, d_in, f"M={M} sampled")
    for m in (0, 255, 256, 511, 512, 1535, 1536, 1791, 1792, M - 1):
        ref_m = oracle.linear(x[m:m + 1], wb, packed, alpha, True)[0]
        _assert_elementwise(y[m], ref_m, xa[m] @ np.abs(weff).T, d_in, f"M={M} row {m}")
