"""GPU parity: bitdelta_linear_grouped (one shared W_base, per-segment variant
ids, variant 0 = base model) against the oracle ("Serving architecture":
base weights shared-read by every variant, the request's model id selects the
delta)."""
import numpy as np
import pytest
import torch

import bit_weight_delta_gb300 as bd
import oracle
import synth
from gpu_util import assert_linear_close, bf16_values, to_dev, to_dev_bf16

pytestmark = pytest.mark.gpu


def _setup(seed, d_out, d_in, n_var, lengths, per_row=True, variants=None):
    wb = synth.base_weight(seed, d_out, d_in)
    scales = synth.variant_scales(seed, n_var)
    packs, alphas = [], []
    for v in range(n_var):
        wf = synth.finetuned_weight(seed, wb, b=float(scales[v]), stream=100 + v)
        p, a, _ = oracle.compress(wb, wf, per_row)
        packs.append(p)
        alphas.append(a)
    off, var = synth.segments(seed, lengths, n_var)
    if variants is not None:
        var = np.asarray(variants, np.int32)
    x = synth.activations(seed, int(off[-1]), d_in)
    return wb, packs, alphas, off, var, x


def _run(wb, packs, alphas, off, var, x, per_row):
    dp = [to_dev(p) for p in packs]
    da = [to_dev(a) for a in alphas]
    pt, at = bd.variant_tables(dp, da, "cuda")
    y = bd.bitdelta_linear_grouped(to_dev_bf16(x), to_dev(off), to_dev(var), to_dev_bf16(wb), pt,
                                   at, n_var=len(packs), max_seg_len=int(np.diff(off).max()),
                                   per_row=per_row)
    assert bd.bitdelta_check_error() == 0
    return bf16_values(y)


@pytest.mark.parametrize("per_row", [True, False])
def test_grouped_small_mixed(per_row):
    """Decode rows and long segments, all variant ids including base."""
    lengths = [1, 1, 3, 40, 1, 2, 300, 1, 16, 17, 5]
    wb, packs, alphas, off, var, x = _setup(11, 200, 512, 4, lengths, per_row)
    var = np.array([0, 1, 2, 3, 4, 0, 2, 1, 3, 0, 4], np.int32)
    y = _run(wb, packs, alphas, off, var, x, per_row)
    ref = oracle.linear_grouped(x, off, var, wb, packs, alphas, per_row)
    assert_linear_close(y, ref)
    for s in range(len(var)):     # every segment on its own scale too
        rows = slice(off[s], off[s + 1])
        assert_linear_close(y[rows], ref[rows], f"segment {s}")


def test_grouped_decode_only_ragged_d_in():
    """All segments short; d_in not a multiple of 128 (byte-wise signs)."""
    lengths = [1] * 20 + [2, 3]
    wb, packs, alphas, off, var, x = _setup(12, 130, 200, 5, lengths)
    y = _run(wb, packs, alphas, off, var, x, True)
    assert_linear_close(y, oracle.linear_grouped(x, off, var, wb, packs, alphas, True))


def test_grouped_empty_segments():
    """Zero-length segments (offsets repeat) at the start, between short and
    long segments and at the end: they produce no rows and no tiles, and the
    rows around them keep their own variants."""
    lengths = [0, 3, 0, 300, 0, 1, 0, 40, 0]
    wb, packs, alphas, off, var, x = _setup(19, 256, 512, 3, lengths,
                                            variants=[2, 1, 3, 2, 1, 3, 2, 1, 3])
    y = _run(wb, packs, alphas, off, var, x, True)
    ref = oracle.linear_grouped(x, off, var, wb, packs, alphas, True)
    assert_linear_close(y, ref)
    for s in range(len(lengths)):
        if lengths[s] > 0:
            rows = slice(off[s], off[s + 1])
            assert_linear_close(y[rows], ref[rows], f"segment {s}")


def test_grouped_long_segments_without_tma_shape():
    """Long segments with d_in % 128 != 0 run through the decode kernel."""
    lengths = [33, 1, 20]
    wb, packs, alphas, off, var, x = _setup(13, 64, 136, 2, lengths)
    y = _run(wb, packs, alphas, off, var, x, True)
    assert_linear_close(y, oracle.linear_grouped(x, off, var, wb, packs, alphas, True))


def test_grouped_base_rows_match_plain_gemm():
    lengths = [5, 300, 1]
    wb, packs, alphas, off, var, x = _setup(14, 256, 512, 2, lengths, variants=[0, 0, 0])
    y = _run(wb, packs, alphas, off, var, x, True)
    ref = (to_dev_bf16(x).float() @ to_dev_bf16(wb).float().T).double().cpu().numpy()
    assert_linear_close(y, ref)


def test_grouped_equals_single_variant_calls():
    lengths = [2, 260, 1, 7]
    wb, packs, alphas, off, var, x = _setup(15, 384, 1024, 3, lengths,
                                            variants=[1, 2, 3, 2])
    y = _run(wb, packs, alphas, off, var, x, True)
    for s in range(4):
        rows = slice(off[s], off[s + 1])
        v = var[s] - 1
        single = bd.bitdelta_linear(to_dev_bf16(x[rows]), to_dev_bf16(wb), to_dev(packs[v]),
                                    to_dev(alphas[v]), per_row=True)
        assert_linear_close(y[rows], bf16_values(single), f"segment {s}")


def test_grouped_bad_variant_id_is_reported():
    """A variant id outside [0, n_var] in device memory: no fault, an error status."""
    lengths = [1, 2]
    wb, packs, alphas, off, var, x = _setup(16, 64, 128, 1, lengths, variants=[0, 5])
    dp = [to_dev(p) for p in packs]
    da = [to_dev(a) for a in alphas]
    pt, at = bd.variant_tables(dp, da, "cuda")
    bd.bitdelta_linear_grouped(to_dev_bf16(x), to_dev(off), to_dev(var), to_dev_bf16(wb), pt, at,
                               n_var=1, max_seg_len=2, per_row=True)
    assert bd.bitdelta_check_error() == 7   # BD_ERR_DEVICE_BOUNDS
    assert bd.bitdelta_check_error() == 0


@pytest.mark.parametrize("per_row", [True, False])
def test_grouped_at_most_eight_short_rows(per_row):
    """At most 8 short rows in the whole batch (here 8 one-row segments that
    alternate two variants, as in a decode step of two tenants): the short
    rows run through the ring with a single token tile."""
    lengths = [1] * 8
    wb, packs, alphas, off, var, x = _setup(17, 320, 1024, 2, lengths, per_row,
                                            variants=[1, 2, 1, 2, 1, 2, 1, 2])
    y = _run(wb, packs, alphas, off, var, x, per_row)
    ref = oracle.linear_grouped(x, off, var, wb, packs, alphas, per_row)
    assert_linear_close(y, ref)
    for s in range(len(var)):
        assert_linear_close(y[s:s + 1], ref[s:s + 1], f"row {s}")


def test_grouped_few_rows_with_base_and_ragged_d_out():
    """Seven short rows (base and three variants) on a d_out that is not a
    multiple of 16: single token tile, partial last row group."""
    lengths = [2, 1, 3, 1]
    wb, packs, alphas, off, var, x = _setup(18, 250, 512, 3, lengths,
                                            variants=[3, 0, 1, 2])
    y = _run(wb, packs, alphas, off, var, x, True)
    ref = oracle.linear_grouped(x, off, var, wb, packs, alphas, True)
    assert_linear_close(y, ref)


def test_grouped_unaligned_sign_rows_take_the_register_pass():
    """d_in % 128 == 0 but one variant's packed signs start 8 bytes past a
    16-byte boundary: groups holding that variant take the register-pipelined
    pass (byte-wise sign loads), the others the ring; both match the oracle."""
    lengths = [1, 3, 1, 2, 1, 5]
    d_out, d_in = 192, 512
    wb, packs, alphas, off, var, x = _setup(19, d_out, d_in, 3, lengths,
                                            variants=[1, 2, 3, 1, 0, 2])
    dp = [to_dev(p) for p in packs]
    raw = torch.empty(packs[1].size + 8, dtype=torch.uint8, device="cuda")
    shifted = raw[8:8 + packs[1].size].view(packs[1].shape)
    shifted.copy_(dp[1])
    assert shifted.data_ptr() % 16 == 8
    dp[1] = shifted
    da = [to_dev(a) for a in alphas]
    pt, at = bd.variant_tables(dp, da, "cuda")
    y = bd.bitdelta_linear_grouped(to_dev_bf16(x), to_dev(off), to_dev(var), to_dev_bf16(wb), pt,
                                   at, n_var=3, max_seg_len=int(np.diff(off).max()), per_row=True)
    assert bd.bitdelta_check_error() == 0
    ref = oracle.linear_grouped(x, off, var, wb, packs, alphas, True)
    assert_linear_close(bf16_values(y), ref)


def test_grouped_more_segments_than_one_tensor_core_launch():
    """1100 segments: the tensor-core kernel holds 1024 in shared memory, so
    the long segments run in two launches (segments 0-1023, 1024-1099), with
    long segments in both slices and short rows between them; every long
    segment is checked at its first, middle and last row, every short row
    whole."""
    n_seg = 1100
    rng = np.random.default_rng(61)
    lengths = [1 + int(rng.integers(0, 3)) for _ in range(n_seg)]
    for s in (5, 700, 1023, 1024, 1050, 1099):
        lengths[s] = 40 + s % 7
    wb, packs, alphas, off, var, x = _setup(61, 256, 256, 3, lengths)
    y = _run(wb, packs, alphas, off, var, x, True)
    rows = []
    for s in range(n_seg):
        a, b = int(off[s]), int(off[s + 1])
        rows.extend([a, (a + b) // 2, b - 1] if b - a > 16 else range(a, b))
    rows = np.array(sorted(set(rows)))
    seg_of = np.searchsorted(off, rows, side="right") - 1
    sub_off = np.arange(len(rows) + 1, dtype=np.int32)
    ref = oracle.linear_grouped(x[rows], sub_off, var[seg_of].astype(np.int32), wb, packs,
                                alphas, True)
    for k, r in enumerate(rows):
        assert_linear_close(y[r], ref[k], f"row {r} (segment {seg_of[k]})")


def test_grouped_short_row_list_limit_refused_before_any_launch():
    """More decode-kernel rows than its shared-memory row list holds: the call
    returns BD_ERR_UNSUPPORTED_SHAPE before launching anything (y keeps its
    contents, the error word stays clear)."""
    n_seg, seg_len, d_out, d_in = 3300, 16, 8, 128
    off = np.arange(n_seg + 1, dtype=np.int32) * seg_len
    var = np.zeros(n_seg, np.int32)
    M = int(off[-1])
    x = torch.zeros((M, d_in), dtype=torch.bfloat16, device="cuda")
    wb = torch.zeros((d_out, d_in), dtype=torch.bfloat16, device="cuda")
    y = torch.full((M, d_out), 7.0, dtype=torch.bfloat16, device="cuda")
    pt, at = bd.variant_tables([], [], "cuda")
    with pytest.raises(bd.BitDeltaError) as err:
        bd.bitdelta_linear_grouped(x, to_dev(off), to_dev(var), wb, pt, at, n_var=0,
                                   max_seg_len=seg_len, per_row=True, out=y)
    assert err.value.code == 2   # BD_ERR_UNSUPPORTED_SHAPE
    torch.cuda.synchronize()
    assert bd.bitdelta_check_error() == 0
    assert bool((y == 7.0).all())
