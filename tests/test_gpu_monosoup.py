"""GPU parity of the MonoSoup merge against the fp64 oracle.

Page "BitDelta: serving 14 Zen models from one GPU cluster", section
"MonoSoup: complementing the single checkpoint with SVD".  Inputs: seeded
checkpoints whose Δ_i are a rank-r signal plus small dense noise (a gap after
σ_r, the structure the page attributes to fine-tuning).

Tolerances.  The GPU forms τ_i by block subspace iteration in fp32.  Its own
algorithmic error with two power iterations on these inputs (σ_r/σ_{r+1} >
40) is below 1e-6 of max|τ| (the subspace error shrinks like
(σ_{r+1}/σ_r)^5); fp32 products over d <= 4096 terms add about
u·sqrt(d)·κ ~ 6e-8·64·4 ~ 1.5e-5.  So the fp32 correction (1/k)·Σ τ_i must
match the oracle within COR_TOL = 1e-4 of its largest magnitude, and every
bf16 element of W_merged must be the rounding (to nearest) of some value
within that same absolute bound of the oracle's fp64 value: its rounding
interval [got − ulp/2, got + ulp/2] must reach [exact − tol, exact + tol].
Where W_base is near zero the bound spans several bf16 ulps of the tiny
result; elsewhere it allows at most the neighbour of the oracle's rounding.
"""
import numpy as np
import pytest
import torch

import bit_weight_delta_gb300 as bd
import oracle
import oracle.monosoup as oms
import synth

pytestmark = pytest.mark.gpu

COR_TOL = 1e-4


def _dev(bits):
    return torch.from_numpy(bits.view(np.int16)).cuda().view(torch.bfloat16)


def _host(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def _check_against_oracle(wb, ws, rank, power_iters=2):
    out_ref, merged_ref, corr_ref = oracle.monosoup_merge(wb, ws, rank)
    wb_d = _dev(wb)
    corr = torch.empty(wb.shape, dtype=torch.float32, device="cuda")
    out = bd.bitdelta_monosoup(wb_d, [_dev(w) for w in ws], rank, power_iters=power_iters,
                               seed=5, correction=corr)
    torch.cuda.synchronize()
    assert bd.bitdelta_check_error() == 0
    c = corr.cpu().numpy().astype(np.float64)
    scale = max(np.abs(corr_ref).max(), 1e-30)
    err = np.abs(c - corr_ref).max() / scale
    assert err <= COR_TOL, f"correction off by {err:.3e} of its max"
    got = _host(out)
    diff = got != out_ref
    if diff.any():
        g = oms.bf16_to_f64(got[diff])
        # bf16 ulp at g: 2^(exponent - 7); the fp32 sum W_base + c adds a
        # relative 2^-24 before the final rounding
        _, e = np.frexp(g)
        half_ulp = np.ldexp(1.0, np.maximum(e, -125) - 9)
        tol = COR_TOL * scale + 2.0**-24 * np.abs(merged_ref[diff])
        assert np.all(np.abs(g - merged_ref[diff]) <= half_ulp + tol)
    return err, int(diff.sum())


@pytest.mark.parametrize("d_out,d_in,rank,k", [
    (256, 512, 8, 3),     # several tiles along both sides
    (200, 520, 5, 2),     # ragged: d_out not a multiple of 64, d_in of 64
    (512, 384, 16, 2),    # d_out > d_in
    (640, 1000, 64, 2),   # the largest rank
    (96, 64, 20, 1),      # one checkpoint, rank padded to 32
    (203, 256, 12, 2),    # d_out not a multiple of 8 (padded rows of V's bf16 terms)
])
def test_merge_matches_oracle(d_out, d_in, rank, k):
    wb = synth.base_weight(d_out + d_in, d_out, d_in)
    ws = synth.monosoup_checkpoints(rank + k, wb, k, rank)
    _check_against_oracle(wb, ws, rank)


def test_rank_zero_returns_the_base():
    wb = synth.base_weight(3, 128, 256)
    ws = synth.monosoup_checkpoints(3, wb, 2, 4)
    corr = torch.full((128, 256), 7.0, dtype=torch.float32, device="cuda")
    out = bd.bitdelta_monosoup(_dev(wb), [_dev(w) for w in ws], 0, correction=corr)
    torch.cuda.synchronize()
    assert np.array_equal(_host(out), wb)
    assert not torch.any(corr)


def test_exactly_low_rank_checkpoints_average():
    # Δ_i = u_i v_iᵀ (integers, rank 1 < r = 4): the merge is the plain
    # average; Y has dependent columns, which the Cholesky step drops
    d_out, d_in, k = 64, 128, 4
    g = np.random.default_rng(9)
    ws = []
    for _ in range(k):
        u = g.integers(-3, 4, d_out).astype(np.float32)
        v = g.integers(-3, 4, d_in).astype(np.float32)
        ws.append(synth.bf16_bits(np.outer(u, v)))
    wb = synth.bf16_bits(np.zeros((d_out, d_in), np.float32))
    out = bd.bitdelta_monosoup(_dev(wb), [_dev(w) for w in ws], 4)
    torch.cuda.synchronize()
    avg = np.mean([synth.bf16_to_f32(w) for w in ws], axis=0)
    got = synth.bf16_to_f32(_host(out))
    nz = avg != 0
    assert np.array_equal(got[nz], avg[nz])
    assert np.all(np.abs(got[~nz]) < 1e-4)


def test_bad_arguments_are_rejected():
    wb = torch.zeros((64, 128), dtype=torch.bfloat16, device="cuda")
    w = torch.zeros_like(wb)
    for kwargs in ({"rank": 65}, {"rank": 65, "power_iters": 2}, {"rank": 4, "power_iters": 17}):
        with pytest.raises(bd.BitDeltaError) as e:
            bd.bitdelta_monosoup(wb, [w], **kwargs)
        assert e.value.code == 2
    small = torch.zeros((16, 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(bd.BitDeltaError) as e:
        bd.bitdelta_monosoup(small, [small.clone()], 20)     # rank > min(d_out, d_in)
    assert e.value.code == 2


def test_full_size_layer_one_checkpoint():
    # one 4096 x 4096 layer (the decode layer's shape), rank 32
    wb = synth.base_weight(41, 4096, 4096)
    ws = synth.monosoup_checkpoints(41, wb, 1, 32)
    err, n_diff = _check_against_oracle(wb, ws, 32)
    assert n_diff < 0.001 * wb.size
