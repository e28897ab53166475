"""GPU parity: cosine similarity of 1-bit task vectors (page section
"K-Merge": pairwise cosine similarity of the requested adapter's task vector
with every pool member, and the most similar member) against the oracle's
element-by-element fp64 definition."""
import numpy as np
import pytest
import torch

import bit_weight_delta_gb300 as bd
import oracle
import synth
import synth.device as sd

pytestmark = pytest.mark.gpu
# Both sides are fp64 and differ only in summation order; the oracle adds up
# to d_out·d_in ≈ 1.2e6 terms one after another, whose rounding bound is about
# n·u·(Σ|terms| / |dot|) ≈ 1.2e6 · 1.1e-16 ≈ 1.4e-10 on the cosine here.
COS_ATOL = 1e-9


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _run(pa, aa, pool, per_row):
    dp = [_dev(p) for p, _ in pool]
    da = [_dev(a) for _, a in pool]
    pt, at = bd.variant_tables(dp, da, "cuda")
    cos, best = bd.bitdelta_sign_similarity(_dev(pa), _dev(aa), pt, at, len(pool), per_row)
    assert bd.bitdelta_check_error() == 0
    return cos.cpu().numpy(), int(best.item())


@pytest.mark.parametrize("per_row", [True, False])
@pytest.mark.parametrize("shape,n_b", [((300, 4096), 5), ((300, 4096), 37), ((77, 136), 6),
                                       ((8, 16), 1)])
def test_similarity_matches_oracle(shape, n_b, per_row):
    d_out, d_in = shape
    rng = np.random.default_rng(d_out + n_b)
    n_alpha = d_out if per_row else 1
    pa = rng.integers(0, 256, (d_out, d_in // 8), dtype=np.uint8)
    aa = rng.uniform(1e-4, 2e-3, n_alpha).astype(np.float32)
    pool = []
    for b in range(n_b):
        # members from near copies of the candidate to independent signs
        flip = rng.random((d_out, d_in // 8, 8)) < (b + 1) / (n_b + 1) * 0.5
        bits = np.unpackbits(pa, axis=1, bitorder="little").reshape(d_out, d_in // 8, 8)
        pb = np.packbits((bits ^ flip).reshape(d_out, d_in), axis=1, bitorder="little")
        pool.append((pb, rng.uniform(1e-4, 2e-3, n_alpha).astype(np.float32)))
    cos, best = _run(pa, aa, pool, per_row)
    ref = np.array([oracle.sign_cosine(pa, aa, pb, ab, per_row)[0] for pb, ab in pool])
    np.testing.assert_allclose(cos, ref, atol=COS_ATOL, rtol=0)
    assert best == int(np.argmax(ref))


def test_identical_and_negated_members():
    rng = np.random.default_rng(1)
    pa = rng.integers(0, 256, (64, 512), dtype=np.uint8)
    aa = rng.uniform(1e-4, 2e-3, 64).astype(np.float32)
    other = rng.integers(0, 256, (64, 512), dtype=np.uint8)
    pool = [(other, aa), (~pa, aa), (pa, aa)]
    cos, best = _run(pa, aa, pool, True)
    assert abs(cos[1] + 1) < COS_ATOL and abs(cos[2] - 1) < COS_ATOL and best == 2


def test_similarity_full_size_grouped_variants():
    """The 14 fine-tuned variants of the grouped workload's 4096->14336 layer:
    variant 1 against the other 13 (per-row α, compressed on the GPU; the
    oracle compresses the same bytes itself)."""
    d_out, d_in, n_var, seed = 14336, 4096, 14, 4
    scales = synth.variant_scales(seed, n_var)
    wb = sd.normal_bf16((d_out, d_in), seed, 100, 0.02)
    packs, alphas, o_packs, o_alphas = [], [], [], []
    wb_h = wb.view(torch.int16).cpu().numpy().view(np.uint16)
    for v in range(n_var):
        wf = sd.finetuned_bf16(wb, seed, 1000 + v, float(scales[v]))
        p, a = bd.bitdelta_compress(wb, wf, per_row=True)
        packs.append(p)
        alphas.append(a)
        op, oa, _ = oracle.compress(wb_h, wf.view(torch.int16).cpu().numpy().view(np.uint16), True)
        o_packs.append(op)
        o_alphas.append(oa)
    pt, at = bd.variant_tables(packs[1:], alphas[1:], "cuda")
    cos, best = bd.bitdelta_sign_similarity(packs[0], alphas[0], pt, at, n_var - 1, True)
    assert bd.bitdelta_check_error() == 0
    best = int(best.item())
    ref = np.array([oracle.sign_cosine(o_packs[0], o_alphas[0], o_packs[b], o_alphas[b], True)[0]
                    for b in range(1, n_var)])
    # the two sides' α agree to 1e-6 relative (the compress bar), so their
    # cosines agree to about twice that
    np.testing.assert_allclose(cos.cpu().numpy(), ref, atol=1e-5, rtol=0)
    assert best == int(np.argmax(ref))
