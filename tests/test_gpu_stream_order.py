"""Stream order across calls, with no synchronisation between them.

The decode kernel of bitdelta_linear ("Serving architecture", fused kernel)
is launched with programmatic dependent launch and issues its first W_base
and sign loads before it waits for the kernel ahead of it; x and α are read
after that wait.  These tests chain calls on one stream the way a serving
step does and check every output against the oracle:

- compress, then a linear over the signs it just wrote (the same buffers
  reused for six fine-tunes): a linear that read signs of the previous
  fine-tune would miss the element-wise bound by far, since each
  fine-tune's delta is as large as the weights;
- reconstruct, then a linear whose W_base is the W_eff it just wrote;
- linears whose x is the previous linear's y (a stack of layers), with the
  y buffers filled with a large constant beforehand, so that reading x
  before the previous layer finished would show.
"""
import numpy as np
import pytest
import torch

import bit_weight_delta_gb300 as bd
import oracle
import synth
from gpu_util import (assert_split_elementwise, bf16_values, from_dev_bf16, to_dev,
                      to_dev_bf16)

pytestmark = pytest.mark.gpu

BIG_B = 0.02


def _assert_split_close(y, x, wb, packed, alpha, per_row, what):
    assert_split_elementwise(y, x, wb, packed, alpha, per_row, what)


@pytest.mark.parametrize("M", [4, 12])
def test_compress_then_linear_on_one_stream(M):
    """M = 4 runs the cp.async ring kernel, M = 12 the register kernel."""
    d_out, d_in, n_ft = 4096, 1024, 6
    wb = synth.base_weight(61, d_out, d_in)
    x = synth.activations(61, M, d_in)
    fts = [synth.finetuned_weight(61, wb, b=BIG_B, stream=300 + i) for i in range(n_ft)]
    wb_d, x_d = to_dev_bf16(wb), to_dev_bf16(x)
    wf_d = [to_dev_bf16(w) for w in fts]
    packed = torch.empty((d_out, d_in // 8), dtype=torch.uint8, device="cuda")
    alpha = torch.empty((d_out,), dtype=torch.float32, device="cuda")
    ys = [torch.empty((M, d_out), dtype=torch.bfloat16, device="cuda") for _ in range(n_ft)]
    torch.cuda.synchronize()
    for i in range(n_ft):
        bd.bitdelta_compress(wb_d, wf_d[i], per_row=True, packed_out=packed, alpha_out=alpha)
        bd.bitdelta_linear(x_d, wb_d, packed, alpha, per_row=True, out=ys[i])
    torch.cuda.synchronize()
    assert bd.bitdelta_check_error() == 0
    for i in range(n_ft):
        p_ref, a_ref = oracle.compress(wb, fts[i], True)[:2]
        _assert_split_close(bf16_values(ys[i]), x, wb, p_ref, a_ref, True, f"fine-tune {i}")


def test_reconstruct_then_linear_over_w_eff():
    """W_eff of each fine-tune written by bitdelta_reconstruct and used at once
    as the base of a linear with α = 0 (so y = x·W_effᵀ)."""
    d_out, d_in, M, n_ft = 4096, 1024, 8, 4
    wb = synth.base_weight(62, d_out, d_in)
    x = synth.activations(62, M, d_in)
    comp = [oracle.compress(wb, synth.finetuned_weight(62, wb, b=BIG_B, stream=310 + i), True)[:2]
            for i in range(n_ft)]
    wb_d, x_d = to_dev_bf16(wb), to_dev_bf16(x)
    pk_d = [to_dev(p) for p, _ in comp]
    al_d = [to_dev(a) for _, a in comp]
    zero_a = torch.zeros((1,), dtype=torch.float32, device="cuda")
    w_eff = torch.empty((d_out, d_in), dtype=torch.bfloat16, device="cuda")
    ys = [torch.empty((M, d_out), dtype=torch.bfloat16, device="cuda") for _ in range(n_ft)]
    torch.cuda.synchronize()
    for i in range(n_ft):
        bd.bitdelta_reconstruct(wb_d, pk_d[i], al_d[i], per_row=True, out=w_eff)
        bd.bitdelta_linear(x_d, w_eff, pk_d[0], zero_a, per_row=False, out=ys[i])
    torch.cuda.synchronize()
    assert bd.bitdelta_check_error() == 0
    for i in range(n_ft):
        weff_ref = oracle.reconstruct(wb, comp[i][0], comp[i][1], True)
        _assert_split_close(bf16_values(ys[i]), x, weff_ref, comp[0][0],
                            np.zeros(1, np.float32), False, f"fine-tune {i}")


@pytest.mark.parametrize("M", [1, 8, 16])
def test_layer_stack_output_feeds_next_input(M):
    """Eight square layers, y_l = linear(y_{l-1}); each layer checked against
    the oracle on the input the GPU actually gave it."""
    d, L = 2048, 8
    layers = []
    for l in range(L):
        wb = synth.base_weight(63 + l, d, d, sigma=1.0 / np.sqrt(d))
        wf = synth.finetuned_weight(63 + l, wb, b=0.01 / np.sqrt(d) * 50, stream=320)
        p, a = oracle.compress(wb, wf, True)[:2]
        layers.append((wb, p, a))
    dev = [(to_dev_bf16(wb), to_dev(p), to_dev(a)) for wb, p, a in layers]
    x0 = synth.activations(63, M, d)
    acts = [to_dev_bf16(x0)] + [torch.full((M, d), 3.0e4, dtype=torch.bfloat16, device="cuda")
                                for _ in range(L)]
    torch.cuda.synchronize()
    for l in range(L):
        wb_d, p_d, a_d = dev[l]
        bd.bitdelta_linear(acts[l], wb_d, p_d, a_d, per_row=True, out=acts[l + 1])
    torch.cuda.synchronize()
    assert bd.bitdelta_check_error() == 0
    for l in range(L):
        wb, p, a = layers[l]
        x_in = from_dev_bf16(acts[l])
        assert np.isfinite(synth.bf16_to_f32(x_in)).all()
        _assert_split_close(bf16_values(acts[l + 1]), x_in, wb, p, a, True, f"layer {l}")
