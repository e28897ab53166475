"""GPU parity at the full benchmark sizes, on sampled outputs the oracle
computes one by one.

Prefill: the four projections of a Llama-70B-sized layer at 2048 tokens
(QKV 8192->10240, O 8192->8192, gate+up 8192->57344, down 28672->8192),
per-row α, run through the tensor-core path the bench times; the oracle
compresses the same W_base/W_ft bytes on the host and computes y for tokens
at tile boundaries over every output column.

Grouped: shared W_base 4096->14336 with 14 fine-tuned variants (Laplace
scales drawn from U[5e-4, 2e-3]), 64 one-row decode segments and four
512-row prefill segments, variant ids uniform over {base, 1..14}; the oracle
checks every decode row and 16 rows of each prefill segment.

Inputs come from the seeded device generator (the generator is shared by both
sides; it holds none of the method's arithmetic).  Page "BitDelta: serving 14
Zen models from one GPU cluster", sections "Mathematical foundation" and
"Serving architecture".
"""
import numpy as np
import pytest
import torch

import bit_weight_delta_gb300 as bd
import oracle
import synth
import synth.device as sd
from gpu_util import assert_linear_close, bf16_values, from_dev_bf16

pytestmark = pytest.mark.gpu

PREFILL_SHAPES = [(10240, 8192), (8192, 8192), (57344, 8192), (8192, 28672)]
TOKENS = 2048
SAMPLED_TOKENS = np.array([0, 1, 255, 256, 1023, 1024, 2046, 2047])


@pytest.mark.parametrize("shape", PREFILL_SHAPES, ids=lambda s: f"{s[0]}x{s[1]}")
def test_prefill_full_size_sampled(shape):
    d_out, d_in = shape
    torch.cuda.set_device(0)
    wb, wf = sd.layer(3, d_out, d_in, stream=1)
    packed, alpha = bd.bitdelta_compress(wb, wf, per_row=True)
    x = sd.normal_bf16((TOKENS, d_in), 3, 5000)
    y = bd.bitdelta_linear(x, wb, packed, alpha, per_row=True)
    assert bd.bitdelta_check_error() == 0
    y_rows = bf16_values(y[torch.from_numpy(SAMPLED_TOKENS).cuda()])
    # oracle: its own compression of the same bytes, then y at the sampled rows
    wb_h, wf_h = from_dev_bf16(wb), from_dev_bf16(wf)
    del wb, wf, packed, alpha, y
    torch.cuda.empty_cache()
    o_packed, o_alpha, _ = oracle.compress(wb_h, wf_h, True)
    del wf_h
    x_h = from_dev_bf16(x[torch.from_numpy(SAMPLED_TOKENS).cuda()])
    ref = oracle.linear(x_h, wb_h, o_packed, o_alpha, True)
    for i, t in enumerate(SAMPLED_TOKENS):
        assert_linear_close(y_rows[i], ref[i], f"{shape} token {t}")


def test_grouped_full_size_sampled():
    d_out, d_in, n_var, seed = 14336, 4096, 14, 4
    torch.cuda.set_device(0)
    scales = synth.variant_scales(seed, n_var)
    off, var = synth.segments(seed, [1] * 64 + [512] * 4, n_var)
    M = int(off[-1])
    wb = sd.normal_bf16((d_out, d_in), seed, 100, 0.02)
    packs, alphas, wfs = [], [], []
    for v in range(n_var):
        wf = sd.finetuned_bf16(wb, seed, 1000 + v, float(scales[v]))
        p, a = bd.bitdelta_compress(wb, wf, per_row=True)
        packs.append(p)
        alphas.append(a)
        wfs.append(from_dev_bf16(wf))
        del wf
    pt, at = bd.variant_tables(packs, alphas, "cuda")
    x = sd.normal_bf16((M, d_in), seed, 77)
    y = bd.bitdelta_linear_grouped(x, torch.from_numpy(off).cuda(), torch.from_numpy(var).cuda(),
                                   wb, pt, at, n_var=n_var, max_seg_len=512, per_row=True)
    assert bd.bitdelta_check_error() == 0
    # rows the oracle checks: every decode row, 16 spread over each prefill segment
    rows = []
    for s in range(len(var)):
        a, b = int(off[s]), int(off[s + 1])
        rows.extend(range(a, b) if b - a == 1 else np.linspace(a, b - 1, 16).astype(int))
    rows = np.array(sorted(set(rows)))
    y_rows = bf16_values(y[torch.from_numpy(rows).cuda()])
    wb_h, x_h = from_dev_bf16(wb), from_dev_bf16(x)
    o_packs, o_alphas = [], []
    for v in range(n_var):
        p, a, _ = oracle.compress(wb_h, wfs[v], True)
        o_packs.append(p)
        o_alphas.append(a)
    # evaluate the sampled rows as one-row segments of their own variant
    seg_of = np.searchsorted(off, rows, side="right") - 1
    sub_off = np.arange(len(rows) + 1, dtype=np.int32)
    ref = oracle.linear_grouped(x_h[rows], sub_off, var[seg_of].astype(np.int32), wb_h, o_packs,
                                o_alphas, True)
    for k, r in enumerate(rows):
        assert_linear_close(y_rows[k], ref[k], f"row {r} (variant {var[seg_of[k]]})")
    assert len(rows) == 64 + 4 * 16
