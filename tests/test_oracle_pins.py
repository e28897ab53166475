"""Pins of the CPU oracle to facts outside itself (no GPU).

Each test ties one oracle function to something the BitDelta page fixes or
the mathematics forces: hand-derived fixtures, closed forms, library routines
(math.fsum, numpy matmul, numpy unpackbits, torch's bf16 cast), exactness
cases and invariants.  Page citations name "BitDelta: serving 14 Zen models
from one GPU cluster" and a section on it.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _val(v):
    if v == "+0":
        return 0.0
    if v == "-0":
        return -0.0
    return float(v)


def _bits(rows):
    a = np.array([[_val(v) for v in r] for r in rows], dtype=np.float32)
    bits = synth.bf16_bits(a)
    # every fixture value is exact in bf16
    assert np.array_equal(synth.bf16_to_f32(bits), a)
    assert np.array_equal(np.signbit(synth.bf16_to_f32(bits)), np.signbit(a))
    return bits


@pytest.fixture(scope="module")
def tiny():
    with open(os.path.join(GOLDEN, "tiny_8x16.json")) as f:
        g = json.load(f)
    g["wb"] = _bits(g["w_base"])
    g["wf"] = _bits(g["w_ft"])
    g["xb"] = _bits(g["x"])
    return g


# ---------------------------------------------------------------- compress

def test_golden_packed_and_alpha_per_row(tiny):
    """Hand-derived 8x16 fixture ("Mathematical foundation", "Infrastructure details")."""
    packed, a32, a64 = oracle.compress(tiny["wb"], tiny["wf"], per_row=True)
    assert packed.tolist() == tiny["packed"]
    assert a32.tolist() == tiny["alpha_per_row"]
    assert a64.tolist() == tiny["alpha_per_row"]


def test_golden_alpha_per_matrix(tiny):
    packed, a32, a64 = oracle.compress(tiny["wb"], tiny["wf"], per_row=False)
    assert packed.tolist() == tiny["packed"]
    assert a32.shape == (1,)
    assert float(a32[0]) == tiny["alpha_per_matrix"]
    assert float(a64[0]) == tiny["alpha_per_matrix"]


def test_packed_size_4096():
    """'Infrastructure details': a 4096x4096 weight packs to 4096x512 bytes."""
    assert oracle.packed_bytes(4096, 4096) == 4096 * 512
    wb, wf = synth.layer(11, 4096, 4096)
    packed, a32, _ = oracle.compress(wb, wf, per_row=True)
    assert packed.shape == (4096, 512) and packed.dtype == np.uint8
    assert a32.shape == (4096,)


def test_storage_arithmetic():
    """'Mathematical foundation' memory arithmetic: 70B bits = 8.75 GB; 140 + 14*8.75 ~ 262 GB; ~87 %."""
    d_in = 8000
    d_out = 70_000_000_000 // d_in
    per_variant = oracle.packed_bytes(d_out, d_in)
    assert per_variant == 8_750_000_000
    total = 140e9 + 14 * per_variant
    assert abs(total / 1e9 - 262.5) < 1e-9
    assert round(1 - total / (14 * 140e9), 2) == 0.87


def test_bit_order_one_hot():
    """One negative delta at (r, c) clears exactly bit c%8 of byte c/8 in row r."""
    d_out, d_in = 3, 24
    wb = synth.bf16_bits(np.full((d_out, d_in), 0.25, np.float32))
    for r in range(d_out):
        for c in range(d_in):
            wf_f = np.full((d_out, d_in), 0.5, np.float32)
            wf_f[r, c] = 0.125
            packed, _, _ = oracle.compress(wb, synth.bf16_bits(wf_f), per_row=True)
            expect = np.full((d_out, d_in // 8), 0xFF, np.uint8)
            expect[r, c // 8] = 0xFF ^ (1 << (c % 8))
            assert np.array_equal(packed, expect), (r, c)


def test_all_positive_all_negative_all_zero():
    wb = synth.bf16_bits(np.full((4, 32), 0.5, np.float32))
    up = synth.bf16_bits(np.full((4, 32), 0.75, np.float32))
    dn = synth.bf16_bits(np.full((4, 32), 0.25, np.float32))
    assert (oracle.compress(wb, up, True)[0] == 0xFF).all()
    assert (oracle.compress(wb, dn, True)[0] == 0x00).all()
    p, a32, _ = oracle.compress(wb, wb, True)          # Δ ≡ 0: sign(0) = +1, α = 0
    assert (p == 0xFF).all() and (a32 == 0).all()


def test_alpha_constant_magnitude_exact():
    """|Δ_ij| ≡ c  =>  α = c exactly, in both scopes ("Mathematical foundation")."""
    for seed in range(4):
        wb, wf, c = synth.constant_magnitude_case(seed)
        _, a_row, _ = oracle.compress(wb, wf, per_row=True)
        _, a_mat, _ = oracle.compress(wb, wf, per_row=False)
        assert (a_row == np.float32(c)).all()
        assert a_mat[0] == np.float32(c)


def test_alpha_matches_exact_sum():
    """α against math.fsum (exactly rounded sum) of |Δ| computed in fp64 from the bf16 inputs."""
    wb, wf = synth.layer(0, 256, 512)
    _, a_row, a_row64 = oracle.compress(wb, wf, per_row=True)
    _, a_mat, a_mat64 = oracle.compress(wb, wf, per_row=False)
    d = np.abs(synth.bf16_to_f32(wf).astype(np.float64) - synth.bf16_to_f32(wb).astype(np.float64))
    for r in range(d.shape[0]):
        exact = math.fsum(d[r].tolist()) / d.shape[1]
        assert abs(a_row64[r] - exact) <= 1e-15 * exact
        assert a_row[r] == np.float32(exact)
    exact = math.fsum(d.ravel().tolist()) / d.size
    assert abs(a_mat64[0] - exact) <= 1e-15 * exact
    assert a_mat[0] == np.float32(exact)


def test_alpha_scopes_are_consistent():
    """Per-matrix α equals the mean of the per-row fp64 means (equal row lengths)."""
    wb, wf = synth.layer(3, 64, 256)
    _, _, r64 = oracle.compress(wb, wf, per_row=True)
    _, _, m64 = oracle.compress(wb, wf, per_row=False)
    assert abs(math.fsum(r64.tolist()) / r64.size - m64[0]) <= 1e-14 * m64[0]


def test_alpha_estimates_laplace_scale():
    """'Mathematical foundation' models Δ ~ Laplace(0, b); E|Δ| = b, so α ≈ b.

    W_ft is rounded to bf16 after adding Δ, which perturbs |Δ| slightly; a few
    per cent is the expected agreement, not a parity bound.
    """
    b = 1e-3
    wb, wf = synth.layer(5, 1024, 1024, b=b)
    _, a, _ = oracle.compress(wb, wf, per_row=False)
    assert abs(a[0] / b - 1) < 0.05


# ---------------------------------------------------------------- reconstruct

def test_golden_reconstruct_per_row(tiny):
    packed = np.array(tiny["packed"], np.uint8)
    alpha = np.array(tiny["alpha_per_row"], np.float32)
    w = oracle.reconstruct(tiny["wb"], packed, alpha, per_row=True)
    # rows whose |Δ| is constant and exactly representable reproduce W_ft
    for r in (0, 1, 2, 4, 5, 7):
        assert np.array_equal(w[r], tiny["wf"][r]), r
    for r, vals in tiny["w_eff_per_row_rows_3_and_6"].items():
        assert np.array_equal(w[int(r)], _bits([vals])[0]), r


def test_golden_reconstruct_per_matrix(tiny):
    packed = np.array(tiny["packed"], np.uint8)
    alpha = np.array([tiny["alpha_per_matrix"]], np.float32)
    w = oracle.reconstruct(tiny["wb"], packed, alpha, per_row=False)
    for key, hexbits in tiny["w_eff_per_matrix_bits"].items():
        r, c = map(int, key.split(","))
        assert int(w[r, c]) == int(hexbits, 16), key


def test_reconstruct_exact_when_constant_magnitude():
    """|Δ| ≡ α with exact bf16 values: W_base + α·sign(Δ) is W_ft bit for bit."""
    for seed in range(6):
        wb, wf, _ = synth.constant_magnitude_case(seed, 8, 16)
        for per_row in (True, False):
            packed, a32, _ = oracle.compress(wb, wf, per_row)
            assert np.array_equal(oracle.reconstruct(wb, packed, a32, per_row), wf)


def test_reconstruct_alpha_zero_is_base():
    """α = 0 returns W_base, except −0 which becomes +0 (IEEE: −0 + +0 = +0)."""
    wb, wf = synth.layer(7, 32, 64)
    wb = wb.copy()
    wb[0, :8] = 0x8000   # −0
    packed, _, _ = oracle.compress(wb, wf, per_row=True)
    w = oracle.reconstruct(wb, packed, np.zeros(32, np.float32), per_row=True)
    expect = wb.copy()
    bits = np.unpackbits(packed, axis=1, bitorder="little").astype(bool)
    # where the bit selects +α = +0, −0 + (+0) = +0; where it selects −α = −0, −0 stays −0
    neg_zero = (wb == 0x8000) & bits
    expect[neg_zero] = 0x0000
    assert np.array_equal(w, expect)


def test_reconstruct_matches_torch_cast():
    """Random layer: oracle W_eff equals torch's fp32 add + RNE bf16 cast, with the
    signs unpacked by numpy (LSB first)."""
    wb, wf = synth.layer(1, 96, 256)
    for per_row in (True, False):
        packed, a32, _ = oracle.compress(wb, wf, per_row)
        bits = np.unpackbits(packed, axis=1, bitorder="little").astype(np.float32)
        a = a32[:, None] if per_row else a32[0]
        s_alpha = torch.from_numpy(np.where(bits > 0, 1.0, -1.0).astype(np.float32) * a)
        w = torch.from_numpy(synth.bf16_to_f32(wb)) + s_alpha
        ref = w.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        assert np.array_equal(oracle.reconstruct(wb, packed, a32, per_row), ref)


def test_bf16_rounding_helper_matches_torch():
    g = np.random.default_rng(0)
    vals = np.concatenate([
        g.standard_normal(20000).astype(np.float32) * np.float32(0.05),
        (1.0 + np.arange(0, 512, dtype=np.float32) * np.float32(2 ** -9)),   # many ties
        np.array([0.0, -0.0, 1e-40, -1e-40, 3.0e38, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8],
                 np.float32),
    ])
    ref = synth.bf16_bits(vals)
    got = np.array([oracle.bf16_round(float(v)) for v in vals], np.uint16)
    assert np.array_equal(got, ref)


# ---------------------------------------------------------------- linear

def test_golden_linear_per_row(tiny):
    packed = np.array(tiny["packed"], np.uint8)
    alpha = np.array(tiny["alpha_per_row"], np.float32)
    y = oracle.linear(tiny["xb"], tiny["wb"], packed, alpha, per_row=True)
    assert y.tolist() == tiny["y_per_row"]


def test_linear_alpha_zero_is_plain_gemm():
    """α = 0 reduces the fused linear to x·W_baseᵀ: numpy matmul in fp64."""
    wb, wf = synth.layer(2, 48, 128)
    x = synth.activations(2, 5, 128)
    packed, _, _ = oracle.compress(wb, wf, True)
    y = oracle.linear(x, wb, packed, np.zeros(48, np.float32), per_row=True)
    ref = synth.bf16_to_f32(x).astype(np.float64) @ synth.bf16_to_f32(wb).astype(np.float64).T
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)


def test_linear_closed_form_popcount():
    """W_base = 0, x = 1: y_n = α_n · (2·popcount(row n) − d_in), exact.

    α values are chosen exact in bf16 so that W_eff = ±α_n exactly."""
    d_out, d_in = 16, 64
    g = np.random.default_rng(3)
    packed = g.integers(0, 256, size=(d_out, d_in // 8), dtype=np.uint8)
    alpha = (g.integers(1, 200, size=d_out) * 2.0 ** -12).astype(np.float32)
    wb = np.zeros((d_out, d_in), np.uint16)
    x = synth.bf16_bits(np.ones((2, d_in), np.float32))
    y = oracle.linear(x, wb, packed, alpha, per_row=True)
    pop = np.array([sum(bin(int(b)).count("1") for b in row) for row in packed])
    ref = alpha.astype(np.float64) * (2 * pop - d_in)
    assert np.array_equal(y[0], ref) and np.array_equal(y[1], ref)


def test_linear_matches_numpy_on_reconstructed():
    """Oracle linear = numpy fp64 matmul of x and the oracle's W_eff."""
    wb, wf = synth.layer(4, 40, 96)
    x = synth.activations(4, 7, 96)
    for per_row in (True, False):
        packed, a32, _ = oracle.compress(wb, wf, per_row)
        weff = oracle.reconstruct(wb, packed, a32, per_row)
        ref = synth.bf16_to_f32(x).astype(np.float64) @ synth.bf16_to_f32(weff).astype(np.float64).T
        np.testing.assert_allclose(oracle.linear(x, wb, packed, a32, per_row), ref,
                                   rtol=1e-12, atol=1e-12)


def test_golden_linear_split_per_row(tiny):
    """The split form on the hand-derived fixture: with per-row α every
    W_base ± α there is exact in bf16 (or α = 0), so the unrounded effective
    weight equals the rounded one and y is the hand-derived y."""
    packed = np.array(tiny["packed"], np.uint8)
    alpha = np.array(tiny["alpha_per_row"], np.float32)
    y = oracle.linear_split(tiny["xb"], tiny["wb"], packed, alpha, per_row=True)
    assert y.tolist() == tiny["y_per_row"]


def test_linear_split_closed_form_popcount():
    """W_base = 0, x = 1: y_n = α_n · (2·popcount(row n) − d_in), exact, for
    any α (nothing is rounded in the split form)."""
    d_out, d_in = 16, 64
    g = np.random.default_rng(13)
    packed = g.integers(0, 256, size=(d_out, d_in // 8), dtype=np.uint8)
    alpha = g.uniform(1e-4, 3e-2, size=d_out).astype(np.float32)
    wb = np.zeros((d_out, d_in), np.uint16)
    x = synth.bf16_bits(np.ones((3, d_in), np.float32))
    y = oracle.linear_split(x, wb, packed, alpha, per_row=True)
    pop = np.array([sum(bin(int(b)).count("1") for b in row) for row in packed])
    ref = alpha.astype(np.float64) * (2 * pop - d_in)
    for m in range(3):
        assert np.array_equal(y[m], ref)
    y1 = oracle.linear_split(x, wb, packed, alpha[:1], per_row=False)
    assert np.array_equal(y1[0], float(alpha[0]) * (2 * pop - d_in))


def test_linear_split_alpha_zero_is_plain_gemm():
    wb, wf = synth.layer(12, 40, 128)
    x = synth.activations(12, 6, 128)
    packed, _, _ = oracle.compress(wb, wf, True)
    y = oracle.linear_split(x, wb, packed, np.zeros(40, np.float32), per_row=True)
    ref = synth.bf16_to_f32(x).astype(np.float64) @ synth.bf16_to_f32(wb).astype(np.float64).T
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)


def test_linear_split_differs_from_rounded_by_the_weight_rounding():
    """The two forms differ only by the bf16 rounding of W_eff: per output,
    |split − rounded| <= Σ_k |x_k| · 2^-8 · |W_eff,k| · (1 + 2^-7) (RNE to 8
    significant bits moves a value by at most 2^-8 of itself), and with
    deltas as large as the weights they do differ."""
    wb = synth.base_weight(14, 32, 256)
    wf = synth.finetuned_weight(14, wb, b=0.02, stream=3)
    x = synth.activations(14, 5, 256)
    for per_row in (True, False):
        packed, a32, _ = oracle.compress(wb, wf, per_row)
        split = oracle.linear_split(x, wb, packed, a32, per_row)
        rounded = oracle.linear(x, wb, packed, a32, per_row)
        weff = synth.bf16_to_f32(oracle.reconstruct(wb, packed, a32, per_row)).astype(np.float64)
        xa = np.abs(synth.bf16_to_f32(x).astype(np.float64))
        bound = 2.0 ** -8 * (1 + 2.0 ** -7) * (xa @ np.abs(weff).T)
        assert (np.abs(split - rounded) <= bound).all()
        assert np.abs(split - rounded).max() > 0


def test_linear_at_matches_full():
    wb, wf = synth.layer(6, 33, 64)
    x = synth.activations(6, 9, 64)
    packed, a32, _ = oracle.compress(wb, wf, True)
    full = oracle.linear(x, wb, packed, a32, True)
    mi = np.repeat(np.arange(9), 33)
    ni = np.tile(np.arange(33), 9)
    at = oracle.linear_at(x, wb, packed, a32, True, mi, ni)
    assert np.array_equal(at, full.ravel())


# ---------------------------------------------------------------- grouped

def _grouped_case(seed=8, d_out=24, d_in=64, n_var=3):
    wb = synth.base_weight(seed, d_out, d_in)
    packs, alphas = [], []
    for v in range(n_var):
        wf = synth.finetuned_weight(seed, wb, b=1e-3 * (v + 1), stream=100 + v)
        p, a, _ = oracle.compress(wb, wf, True)
        packs.append(p)
        alphas.append(a)
    lengths = [1, 3, 1, 5, 2, 1]
    off = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    var = np.array([0, 1, 2, 3, 1, 0], np.int32)
    x = synth.activations(seed, int(off[-1]), d_in)
    return x, off, var, wb, packs, alphas


def test_grouped_equals_per_segment_linear():
    x, off, var, wb, packs, alphas = _grouped_case()
    y = oracle.linear_grouped(x, off, var, wb, packs, alphas, True)
    for s in range(len(var)):
        rows = slice(off[s], off[s + 1])
        if var[s] == 0:
            ref = synth.bf16_to_f32(x[rows]).astype(np.float64) @ \
                synth.bf16_to_f32(wb).astype(np.float64).T
            np.testing.assert_allclose(y[rows], ref, rtol=1e-12, atol=1e-12)
        else:
            v = var[s] - 1
            ref = oracle.linear(x[rows], wb, packs[v], alphas[v], True)
            assert np.array_equal(y[rows], ref)


def test_grouped_empty_segments_change_nothing():
    """Zero-length segments (repeated offsets) inserted anywhere leave every
    row's output as it was without them."""
    x, off, var, wb, packs, alphas = _grouped_case()
    y = oracle.linear_grouped(x, off, var, wb, packs, alphas, True)
    lengths = np.diff(off)
    ins_len, ins_var = [0], [2]
    for L, v in zip(lengths, var):
        ins_len += [int(L), 0]
        ins_var += [int(v), 3]
    off2 = np.concatenate([[0], np.cumsum(ins_len)]).astype(np.int32)
    y2 = oracle.linear_grouped(x, off2, np.array(ins_var, np.int32), wb, packs, alphas, True)
    assert np.array_equal(y, y2)


def test_grouped_at_matches_full():
    x, off, var, wb, packs, alphas = _grouped_case()
    y = oracle.linear_grouped(x, off, var, wb, packs, alphas, True)
    M, N = y.shape
    mi = np.repeat(np.arange(M), N)
    ni = np.tile(np.arange(N), M)
    at = oracle.linear_grouped_at(x, off, var, wb, packs, alphas, True, mi, ni)
    assert np.array_equal(at, y.ravel())


# ------------------------------------------------------------ K-Merge cosine
# Page section "K-Merge": cosine similarity of task vectors; here of their
# 1-bit form α ⊙ S (per-row α).


def test_sign_cosine_hand_example():
    """Two rows of 8 columns worked by hand: row 0 agrees on 7 of 8 signs
    (Σ s_a·s_b = 6), row 1 on 4 of 8 (Σ = 0); α_a = (1/2, 1/4), α_b = (1, 2):
    dot = 1/2·1·6 = 3, |a|² = 8/4 + 8/16 = 2.5, |b|² = 8 + 32 = 40,
    cos = 3 / √100 = 0.3."""
    pa = np.array([[0b10110010], [0xFF]], np.uint8)
    pb = np.array([[0b10010010], [0x0F]], np.uint8)
    cos, dot, na, nb = oracle.sign_cosine(pa, np.array([0.5, 0.25], np.float32), pb,
                                          np.array([1.0, 2.0], np.float32), True)
    assert (dot, na, nb) == (3.0, 2.5, 40.0)
    assert cos == pytest.approx(0.3, abs=1e-15)


def test_sign_cosine_identical_negated_and_symmetric():
    rng = np.random.default_rng(5)
    pa = rng.integers(0, 256, (12, 6), dtype=np.uint8)
    pb = rng.integers(0, 256, (12, 6), dtype=np.uint8)
    aa = rng.uniform(1e-4, 2e-3, 12).astype(np.float32)
    ab = rng.uniform(1e-4, 2e-3, 12).astype(np.float32)
    assert oracle.sign_cosine(pa, aa, pa, aa, True)[0] == pytest.approx(1.0, abs=1e-15)
    assert oracle.sign_cosine(pa, aa, ~pa, aa, True)[0] == pytest.approx(-1.0, abs=1e-15)
    c1 = oracle.sign_cosine(pa, aa, pb, ab, True)[0]
    c2 = oracle.sign_cosine(pb, ab, pa, aa, True)[0]
    assert c1 == c2 and -1.0 <= c1 <= 1.0
    # a common scale of one side's α (a power of two: exact in fp32) does not
    # change the cosine
    assert oracle.sign_cosine(pa, aa, pb, 4 * ab, True)[0] == pytest.approx(c1, rel=1e-12)


def test_sign_cosine_per_matrix_is_the_sign_agreement():
    """With one α per matrix the cosine is (agreements − disagreements)/n,
    counted here with numpy's unpackbits, whatever the two α values."""
    rng = np.random.default_rng(6)
    pa = rng.integers(0, 256, (9, 4), dtype=np.uint8)
    pb = rng.integers(0, 256, (9, 4), dtype=np.uint8)
    ua, ub = np.unpackbits(pa, bitorder="little"), np.unpackbits(pb, bitorder="little")
    agree = int((ua == ub).sum())
    want = (2 * agree - ua.size) / ua.size
    got = oracle.sign_cosine(pa, np.array([7e-4], np.float32), pb, np.array([2e-3], np.float32),
                             False)[0]
    assert got == pytest.approx(want, abs=1e-15)
