"""GPU parity on the 40-layer slice of a Llama-70B-shaped decoder: the same
seeded weights, variants and inputs the slice benchmark draws, the same
library calls, checked against the oracle.

* Decode rows, one full layer (layer 0, all four projections QKV
  8192->10240, O 8192->8192, gate+up 8192->57344, down 28672->8192): the
  batch of 8 rows alternating variants 1, 2, 1, 2, ... as eight one-row
  segments of the grouped linear over the shared W_base; the oracle
  compresses both variants from the same bytes and computes every output of
  every row (the linear bar per row and over the batch).
* Prefill, layer 0: 512 tokens of variant 1 through the tensor-core path;
  the oracle computes every output of tokens at the 256-token tile edges.
* Per-layer compression of the third variant on layers 0 and 39: packed signs
  bit for bit, α within 1e-6 of the oracle's fp64 mean |Δ|.

Page "BitDelta: serving 14 Zen models from one GPU cluster", sections
"Mathematical foundation" (Δ, sign, α = mean|Δ|) and "Serving architecture"
(shared base weights, each request's variant through the fused kernel).
"""
import numpy as np
import pytest
import torch

import bit_weight_delta_gb300 as bd
import oracle
import synth.device as sd
from gpu_util import ALPHA_RTOL, assert_linear_close, bf16_values, from_dev_bf16

pytestmark = pytest.mark.gpu

PROJ_IDS = [s[0] for s in sd.SLICE_SHAPES]
PREFILL_TOKENS = np.array([0, 1, 255, 256, 257, 383, 510, 511])


@pytest.mark.parametrize("proj", range(len(sd.SLICE_SHAPES)), ids=PROJ_IDS)
def test_slice_layer0_decode_rows_and_prefill(proj):
    torch.cuda.set_device(0)
    name, d_out, d_in = sd.SLICE_SHAPES[proj]
    wb = sd.slice_base(0, proj)
    packs, alphas, host_ft = [], [], []
    for v in (1, 2):
        wf = sd.slice_finetuned(wb, 0, proj, v)
        p, a = bd.bitdelta_compress(wb, wf, per_row=True)
        packs.append(p)
        alphas.append(a)
        host_ft.append(from_dev_bf16(wf))
        del wf
    pt, at = bd.variant_tables(packs, alphas, "cuda")
    rows = sd.SLICE_DECODE_ROWS
    xd = sd.slice_inputs(d_in, rows, True)
    off = np.arange(rows + 1, dtype=np.int32)
    var = np.array([1 + (r % 2) for r in range(rows)], np.int32)
    yd = bd.bitdelta_linear_grouped(xd, torch.from_numpy(off).cuda(), torch.from_numpy(var).cuda(),
                                    wb, pt, at, n_var=2, max_seg_len=1, per_row=True)
    xp = sd.slice_inputs(d_in, sd.SLICE_PREFILL_TOKENS, False)
    yp = bd.bitdelta_linear(xp, wb, packs[0], alphas[0], per_row=True)
    assert bd.bitdelta_check_error() == 0
    yd_h = bf16_values(yd)
    yp_h = bf16_values(yp[torch.from_numpy(PREFILL_TOKENS).cuda()])
    wb_h, xd_h = from_dev_bf16(wb), from_dev_bf16(xd)
    xp_h = from_dev_bf16(xp[torch.from_numpy(PREFILL_TOKENS).cuda()])
    del wb, packs, alphas, pt, at, yd, yp, xp
    torch.cuda.empty_cache()

    o_packs, o_alphas = [], []
    for wf_h in host_ft:
        p, a, _ = oracle.compress(wb_h, wf_h, True)
        o_packs.append(p)
        o_alphas.append(a)
    del host_ft
    ref_d = oracle.linear_grouped(xd_h, off, var, wb_h, o_packs, o_alphas, True)
    assert_linear_close(yd_h, ref_d, f"{name} decode batch")
    for r in range(rows):
        assert_linear_close(yd_h[r], ref_d[r], f"{name} decode row {r} (variant {var[r]})")
    ref_p = oracle.linear(xp_h, wb_h, o_packs[0], o_alphas[0], True)
    for i, t in enumerate(PREFILL_TOKENS):
        assert_linear_close(yp_h[i], ref_p[i], f"{name} prefill token {t}")


@pytest.mark.parametrize("proj", range(len(sd.SLICE_SHAPES)), ids=PROJ_IDS)
@pytest.mark.parametrize("layer", [0, 39])
def test_slice_compress_third_variant(layer, proj):
    torch.cuda.set_device(0)
    name, d_out, d_in = sd.SLICE_SHAPES[proj]
    wb = sd.slice_base(layer, proj)
    wf = sd.slice_finetuned(wb, layer, proj, 3)
    packed = torch.empty((d_out, d_in // 8), dtype=torch.uint8, device="cuda")
    alpha = torch.empty((d_out,), dtype=torch.float32, device="cuda")
    bd.bitdelta_compress(wb, wf, per_row=True, packed_out=packed, alpha_out=alpha)
    assert bd.bitdelta_check_error() == 0
    p_gpu, a_gpu = packed.cpu().numpy(), alpha.cpu().numpy().astype(np.float64)
    wb_h, wf_h = from_dev_bf16(wb), from_dev_bf16(wf)
    del wb, wf, packed, alpha
    torch.cuda.empty_cache()
    p_ref, _, a64 = oracle.compress(wb_h, wf_h, True)
    assert np.array_equal(p_gpu, p_ref), f"layer {layer} {name}: packed signs differ"
    rel = np.abs(a_gpu - a64) / np.abs(a64)
    assert rel.max() <= ALPHA_RTOL, f"layer {layer} {name}: alpha rel err {rel.max():.3e}"
