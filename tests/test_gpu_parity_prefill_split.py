"""GPU parity of the prefill kernel's split schedule (bitdelta_linear_ws)
against the oracle.

Page section "Serving architecture": y = x·(W_base + α·unpack(bits))ᵀ with
W_eff built on chip.  With a workspace and a small last round of tiles (at
most a quarter of the device's 76 CTA pairs), that round and the one before
it are cut by k-blocks over the pairs; a tile shared by two pairs is the sum
of their fp32 partials.  A
partial lost, counted twice, stored to the wrong slot or summed from a stale
slot shifts y by the products of a whole k range, far beyond the element-wise
bound used here (the bound of the prefill tile tests: bf16 output rounding
plus a generous fp32 accumulation term).
"""
import numpy as np
import pytest
import torch

import bit_weight_delta_gb300 as bd
import oracle
import synth
from gpu_util import bf16_values, to_dev, to_dev_bf16

pytestmark = pytest.mark.gpu

BIG_B = 0.02


def _layer(seed, d_out, d_in, per_row):
    wb = synth.base_weight(seed, d_out, d_in)
    wf = synth.finetuned_weight(seed, wb, b=BIG_B, stream=2)
    packed, alpha = oracle.compress(wb, wf, per_row)[:2]
    return wb, packed, alpha


def _workspace(M, d_out, d_in):
    need = bd.bitdelta_linear_workspace_bytes(M, d_out, d_in)
    assert need > 0
    return torch.zeros(need, dtype=torch.uint8, device="cuda")


def _run(x, wb, packed, alpha, per_row, ws):
    return bf16_values(bd.bitdelta_linear_ws(to_dev_bf16(x), to_dev_bf16(wb), to_dev(packed),
                                             to_dev(alpha), ws, per_row=per_row))


def _check_all(y, x, wb, packed, alpha, per_row, what):
    d_in = x.shape[1]
    ref = oracle.linear(x, wb, packed, alpha, per_row)
    weff = synth.bf16_to_f32(oracle.reconstruct(wb, packed, alpha, per_row)).astype(np.float64)
    absmag = np.abs(synth.bf16_to_f32(x).astype(np.float64)) @ np.abs(weff).T
    bound = 2.0 ** -8 * np.abs(ref) + d_in * 2.0 ** -22 * absmag
    err = np.abs(y - ref)
    bad = err > bound
    assert not bad.any(), (f"{what}: {int(bad.sum())} outputs off, worst "
                           f"{float((err - bound).max()):.3e} over the bound")


@pytest.fixture
def wide():
    """The split schedule runs on 512-token tiles: force them, so that the
    cases below split whatever the automatic width would pick."""
    bd.bitdelta_set_prefill_tile(512)
    yield
    bd.bitdelta_set_prefill_tile("auto")


@pytest.mark.parametrize("M,d_out,d_in,per_row", [
    (2048, 256 * 40, 256, True),    # 160 tiles on 76 pairs: a round of whole tiles, then
                                    # 84 split in four token-tile groups
    (2000, 256 * 40, 256, False),   # ragged last token tile of every row tile
    (1100, 6902, 1024, True),       # 81 tiles, all split in one group (3 token tiles);
                                    # 76-token last tiles (one MMA), last row tile partly
                                    # past d_out
    (1536, 256 * 53, 384, True),    # 159 tiles: two rounds, then 83 split
])
def test_split_elementwise(M, d_out, d_in, per_row, wide):
    wb, packed, alpha = _layer(31, d_out, d_in, per_row)
    x = synth.activations(31, M, d_in)
    y = _run(x, wb, packed, alpha, per_row, _workspace(M, d_out, d_in))
    assert bd.bitdelta_check_error() == 0
    _check_all(y, x, wb, packed, alpha, per_row, f"M={M} d_out={d_out} d_in={d_in}")


def test_split_deterministic_and_reusable(wide):
    """The partials are summed in k order by whichever contributor finishes
    last: two calls give identical bits, also with a workspace left dirty by
    a call of another shape (the call clears its counters itself)."""
    M, d_out, d_in = 2048, 256 * 40, 256
    wb, packed, alpha = _layer(32, d_out, d_in, True)
    x = synth.activations(32, M, d_in)
    ws = _workspace(M, d_out, d_in)
    a = _run(x, wb, packed, alpha, True, ws)
    wb2, packed2, alpha2 = _layer(33, 6902, 1024, True)
    x2 = synth.activations(33, 1100, 1024)
    _run(x2, wb2, packed2, alpha2, True, ws)
    b = _run(x, wb, packed, alpha, True, ws)
    assert bd.bitdelta_check_error() == 0
    assert np.array_equal(a, b)


def test_split_close_to_unsplit(wide):
    """Only the tiles shared by two pairs change their fp32 sum order (by a
    few fp32 ulps of the partial sums): the split and unsplit calls agree to
    the last bf16 bit on nearly every output."""
    M, d_out, d_in = 2048, 256 * 40, 256
    wb, packed, alpha = _layer(34, d_out, d_in, True)
    x = synth.activations(34, M, d_in)
    a = _run(x, wb, packed, alpha, True, _workspace(M, d_out, d_in))
    b = bf16_values(bd.bitdelta_linear(to_dev_bf16(x), to_dev_bf16(wb), to_dev(packed),
                                       to_dev(alpha), per_row=True))
    assert bd.bitdelta_check_error() == 0
    diff = a != b
    assert diff.mean() < 0.02, f"{int(diff.sum())} of {diff.size} outputs differ"


def test_workspace_errors():
    M, d_out, d_in = 2048, 1024, 256
    wb, packed, alpha = _layer(35, d_out, d_in, True)
    x = synth.activations(35, M, d_in)
    need = bd.bitdelta_linear_workspace_bytes(M, d_out, d_in)
    small = torch.zeros(need - 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(bd.BitDeltaError) as e:
        _run(x, wb, packed, alpha, True, small)
    assert e.value.code == 4   # BD_ERR_WORKSPACE
    big = torch.zeros(need + 512, dtype=torch.uint8, device="cuda")
    with pytest.raises(bd.BitDeltaError) as e:
        _run(x, wb, packed, alpha, True, big[16:])
    assert e.value.code == 3   # BD_ERR_MISALIGNED
    # decode-size calls never split: no workspace needed, one given is ignored
    assert bd.bitdelta_linear_workspace_bytes(16, d_out, d_in) == 0
    y = _run(x[:16], wb, packed, alpha, True, small)
    ref = oracle.linear(x[:16], wb, packed, alpha, True)
    assert np.abs(y - ref).max() <= 1e-2 * np.abs(ref).max()
    assert bd.bitdelta_check_error() == 0
