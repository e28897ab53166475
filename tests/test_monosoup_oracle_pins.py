"""Pins of the MonoSoup oracle to facts outside itself (no GPU).

Page "BitDelta: serving 14 Zen models from one GPU cluster", section
"MonoSoup: complementing the single checkpoint with SVD": W_merged =
W_base + (1/k)·Σ_i τ_i with τ_i the rank-r truncated SVD of Δ_i = W_i −
W_base.  Each test fixes a result by a route that does not reuse the oracle's
own formula: exactly low-rank checkpoints (the merge reduces to the plain
average), a hand-built diagonal case with known singular vectors, the
Eckart-Young residual against a different LAPACK routine (symmetric
eigenvalues), invariances, the rank extremes, and torch's bf16 rounding.
"""
import numpy as np
import pytest
import torch

import oracle
import oracle.monosoup as oms
import synth


def _bits(a):
    bits = synth.bf16_bits(np.asarray(a, dtype=np.float32))
    assert np.array_equal(synth.bf16_to_f32(bits), np.asarray(a, dtype=np.float32))
    return bits


def test_bf16_rne_matches_torch_and_breaks_ties_to_even():
    g = np.random.default_rng(7)
    x = (g.standard_normal(20000) * np.exp(g.uniform(-30, 30, 20000))).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(oms.bf16_rne(x.astype(np.float64)), ref)
    # ties in [1, 2) (bf16 spacing 2^-7): 1 + 2^-8 -> 1.0, 1 + 3·2^-8 -> 1 + 2^-6
    got = oms.bf16_to_f64(oms.bf16_rne(np.array([1 + 2**-8, 1 + 3 * 2**-8, -(1 + 2**-8)])))
    assert got.tolist() == [1.0, 1 + 2**-6, -1.0]


def test_exactly_low_rank_checkpoints_merge_to_their_average():
    # Δ_i = u_i v_iᵀ with small integers: rank 1 <= r, so τ_i = Δ_i and the
    # merge is W_base + mean Δ_i = mean W_i (here W_base = 0).
    d_out, d_in, k = 6, 10, 4
    g = np.random.default_rng(3)
    ws = []
    for _ in range(k):
        u = g.integers(-3, 4, d_out).astype(np.float64)
        v = g.integers(-3, 4, d_in).astype(np.float64)
        ws.append(_bits(np.outer(u, v)))
    wb = _bits(np.zeros((d_out, d_in)))
    merged_bits, merged, corr = oracle.monosoup_merge(wb, ws, rank=2)
    avg = np.mean([synth.bf16_to_f32(w).astype(np.float64) for w in ws], axis=0)
    assert np.allclose(merged, avg, rtol=0, atol=1e-12)
    # multiples of 1/4 below 2^6 are exact in bf16; where the average is 0 the
    # SVD's fp64 rounding residue (~1e-16) is itself a (tiny) bf16 value
    nz = avg != 0
    assert np.array_equal(merged_bits[nz], _bits(avg)[nz])
    assert np.all(np.abs(synth.bf16_to_f32(merged_bits[~nz])) < 1e-12)


def test_signed_permutation_of_a_diagonal():
    # Δ = P·D·Q with D = diag(3, 2, 1, 0.5) in a 5x7 frame and P, Q signed
    # permutations: its singular values are 3, 2, 1, 0.5 and the rank-2
    # truncation keeps exactly the 3 and the 2 at their permuted places.
    d = np.zeros((5, 7))
    for i, s in enumerate([3.0, 2.0, 1.0, 0.5]):
        d[i, i] = s
    p = np.eye(5)[[3, 0, 4, 1, 2]] * np.array([1, -1, 1, 1, -1])[:, None]
    q = np.eye(7)[[6, 2, 0, 5, 1, 3, 4]] * np.array([-1, 1, 1, -1, 1, 1, 1])[:, None]
    delta = p @ d @ q
    keep = np.zeros((5, 7))
    keep[0, 0], keep[1, 1] = 3.0, 2.0
    expect = p @ keep @ q
    wb = _bits(np.zeros((5, 7)))
    merged_bits, merged, _ = oracle.monosoup_merge(wb, [_bits(delta)], rank=2)
    assert np.allclose(merged, expect, rtol=0, atol=1e-12)
    nz = expect != 0
    assert np.array_equal(merged_bits[nz], _bits(expect)[nz])


def test_eckart_young_residual_and_rank():
    g = np.random.default_rng(11)
    delta = g.laplace(0.0, 1e-3, size=(40, 64))
    r = 5
    tau = oms.truncated_svd(delta, r)
    lam = np.sort(np.linalg.eigvalsh(delta @ delta.T))[::-1]      # σ_j², a different routine
    resid = np.sum((delta - tau) ** 2)
    assert resid == pytest.approx(np.sum(lam[r:]), rel=1e-9)
    lam_tau = np.sort(np.linalg.eigvalsh(tau @ tau.T))[::-1]
    assert np.allclose(lam_tau[:r], lam[:r], rtol=1e-9)
    assert np.all(np.abs(lam_tau[r:]) < 1e-12 * lam[0])


def test_identical_checkpoints_and_order():
    wb = synth.base_weight(5, 24, 32)
    ws = synth.monosoup_checkpoints(5, wb, k=3, rank=4)
    _, m1, _ = oracle.monosoup_merge(wb, [ws[0]], rank=4)
    _, m3, _ = oracle.monosoup_merge(wb, [ws[0]] * 3, rank=4)
    assert np.allclose(m1, m3, rtol=0, atol=1e-15)
    _, a, _ = oracle.monosoup_merge(wb, ws, rank=4)
    _, b, _ = oracle.monosoup_merge(wb, ws[::-1], rank=4)
    assert np.allclose(a, b, rtol=0, atol=1e-15)


def test_rank_extremes():
    wb = synth.base_weight(6, 16, 24)
    ws = synth.monosoup_checkpoints(6, wb, k=2, rank=3)
    bits0, m0, c0 = oracle.monosoup_merge(wb, ws, rank=0)
    assert np.array_equal(bits0, wb) and not np.any(c0)
    _, mfull, _ = oracle.monosoup_merge(wb, ws, rank=16)
    base = synth.bf16_to_f32(wb).astype(np.float64)
    mean_delta = np.mean([synth.bf16_to_f32(w).astype(np.float64) - base for w in ws], axis=0)
    assert np.allclose(mfull, base + mean_delta, rtol=0, atol=1e-15)


def test_synthetic_checkpoints_have_a_gap_after_rank_r():
    # the input recipe's premise: a clear gap between σ_r and σ_{r+1}
    wb = synth.base_weight(7, 256, 512)
    r = 8
    w = synth.monosoup_checkpoints(7, wb, k=1, rank=r)[0]
    delta = synth.bf16_to_f32(w).astype(np.float64) - synth.bf16_to_f32(wb)
    s = np.linalg.svd(delta, compute_uv=False)
    assert s[r - 1] > 5 * s[r]
