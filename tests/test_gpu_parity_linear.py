"""GPU parity: bitdelta_linear (decode kernel and tensor-core kernel) against
the oracle: max|y − y_ref| <= 1e-2 · max|y_ref|, fp32 accumulation.

Page section "Serving architecture": the conceptual fused_bitdelta_linear is
F.linear(x, W_base + α·unpack(bits)); the oracle computes it in fp64 with
the bf16-rounded W_eff."""
import numpy as np
import pytest

import bit_weight_delta_gb300 as bd
import oracle
import synth
from gpu_util import assert_linear_close, bf16_values, to_dev_bf16

pytestmark = pytest.mark.gpu


def _layer(seed, d_out, d_in, per_row):
    wb, wf = synth.layer(seed, d_out, d_in)
    packed, alpha = oracle.compress(wb, wf, per_row)[:2]
    return wb, packed, alpha


def _run(x, wb, packed, alpha, per_row):
    return bd.bitdelta_linear(to_dev_bf16(x), to_dev_bf16(wb), bd_tensor(packed),
                              bd_tensor(alpha), per_row=per_row)


def bd_tensor(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


@pytest.mark.parametrize("M", [1, 2, 3, 4, 8, 9, 13, 16])
@pytest.mark.parametrize("per_row", [True, False])
def test_decode_tiny_config(M, per_row):
    """256x512 layer (the tiny config), all decode row counts incl. ragged."""
    wb, packed, alpha = _layer(0, 256, 512, per_row)
    x = synth.activations(0, M, 512)
    y = _run(x, wb, packed, alpha, per_row)
    assert bd.bitdelta_check_error() == 0
    assert_linear_close(bf16_values(y), oracle.linear(x, wb, packed, alpha, per_row), f"M={M}")


@pytest.mark.parametrize("M", [1, 2, 4, 8, 16])
def test_decode_4096(M):
    """The decode sweep layer: 4096x4096, per-row α, M in {1,2,4,8,16}."""
    wb, packed, alpha = _layer(1, 4096, 4096, True)
    x = synth.activations(1, M, 4096)
    y = _run(x, wb, packed, alpha, True)
    assert_linear_close(bf16_values(y), oracle.linear(x, wb, packed, alpha, True), f"M={M}")


@pytest.mark.parametrize("shape", [(8, 16), (37, 136), (130, 1032), (5, 8), (257, 200)])
@pytest.mark.parametrize("M", [1, 7, 16, 40])
def test_ragged_shapes(shape, M):
    """d_out not a multiple of 16, d_in not a multiple of 128 (byte-wise sign
    loads and the 32-column tail); M > 16 with such d_in runs the decode
    kernel over 16-row chunks."""
    d_out, d_in = shape
    wb, packed, alpha = _layer(2, d_out, d_in, True)
    x = synth.activations(2, M, d_in)
    y = _run(x, wb, packed, alpha, True)
    assert_linear_close(bf16_values(y), oracle.linear(x, wb, packed, alpha, True),
                        f"{shape} M={M}")


@pytest.mark.parametrize("M", [17, 256, 300, 513])
@pytest.mark.parametrize("per_row", [True, False])
def test_tensor_core_path(M, per_row):
    """M > 16 with d_in % 128 == 0: tcgen05 kernel.  d_out = 384 spans three
    row tiles; M = 300 and 513 leave ragged token tiles."""
    wb, packed, alpha = _layer(3, 384, 512, per_row)
    x = synth.activations(3, M, 512)
    y = _run(x, wb, packed, alpha, per_row)
    assert bd.bitdelta_check_error() == 0
    assert_linear_close(bf16_values(y), oracle.linear(x, wb, packed, alpha, per_row), f"M={M}")


def test_tensor_core_ragged_d_out_and_long_k():
    """d_out = 200 (partial row tile), d_in = 2048 (32 K-blocks, ring wrap)."""
    wb, packed, alpha = _layer(4, 200, 2048, True)
    x = synth.activations(4, 270, 2048)
    y = _run(x, wb, packed, alpha, True)
    assert_linear_close(bf16_values(y), oracle.linear(x, wb, packed, alpha, True))


def test_tensor_core_many_tiles():
    """More tiles than SMs (persistent loop, both accumulator buffers)."""
    wb, packed, alpha = _layer(5, 4096, 1024, True)
    x = synth.activations(5, 1024, 1024)
    y = bf16_values(_run(x, wb, packed, alpha, True))
    rng = np.random.default_rng(0)
    mi = rng.integers(0, 1024, 4000)
    ni = rng.integers(0, 4096, 4000)
    ref = oracle.linear_at(x, wb, packed, alpha, True, mi, ni)
    assert_linear_close(y[mi, ni], ref)
    # whole rows at the start, middle and end
    for m in (0, 511, 1023):
        assert_linear_close(y[m], oracle.linear(x[m:m + 1], wb, packed, alpha, True)[0])


@pytest.mark.parametrize("d_in", [128, 384, 640])
def test_tensor_core_k_blocks_and_tile_wrap(d_in):
    """K-block counts of 2, 6 and 10 (not multiples of the transform's
    warpgroup count, so a warpgroup's stages cross tile boundaries at varying
    k-blocks) with 2 x 80 tiles: more tiles than SMs, some CTAs take two."""
    d_out, M = 128 * 80, 300
    wb, packed, alpha = _layer(8, d_out, d_in, True)
    x = synth.activations(8, M, d_in)
    y = bf16_values(_run(x, wb, packed, alpha, True))
    assert bd.bitdelta_check_error() == 0
    rng = np.random.default_rng(d_in)
    mi = rng.integers(0, M, 3000)
    ni = rng.integers(0, d_out, 3000)
    assert_linear_close(y[mi, ni], oracle.linear_at(x, wb, packed, alpha, True, mi, ni))
    for m in (0, 255, 256, 299):
        assert_linear_close(y[m], oracle.linear(x[m:m + 1], wb, packed, alpha, True)[0],
                            f"row {m}")


def test_alpha_zero_is_plain_gemm():
    """α = 0: the fused linear is x·W_baseᵀ; compare with torch's cuBLAS GEMM."""
    import torch
    wb, packed, _ = _layer(6, 256, 1024, True)
    alpha = np.zeros(256, np.float32)
    for M in (4, 300):
        x = synth.activations(6, M, 1024)
        y = _run(x, wb, packed, alpha, True)
        ref = (to_dev_bf16(x).float() @ to_dev_bf16(wb).float().T).double().cpu().numpy()
        assert_linear_close(bf16_values(y), ref, f"M={M}")


def test_closed_form_popcount():
    """W_base = 0, x = 1: y_n = α_n·(2·popcount(row n) − d_in)."""
    d_out, d_in = 64, 256
    rng = np.random.default_rng(7)
    packed = rng.integers(0, 256, size=(d_out, d_in // 8), dtype=np.uint8)
    alpha = (rng.integers(1, 200, size=d_out) * 2.0 ** -12).astype(np.float32)
    wb = np.zeros((d_out, d_in), np.uint16)
    pop = np.array([sum(bin(int(b)).count("1") for b in row) for row in packed])
    ref = alpha.astype(np.float64) * (2 * pop - d_in)
    for M in (1, 16, 40):
        x = synth.bf16_bits(np.ones((M, d_in), np.float32))
        y = bf16_values(_run(x, wb, packed, alpha, True))
        assert_linear_close(y, np.tile(ref, (M, 1)), f"M={M}")


def test_wait_timeout_is_reported():
    """A bounded device wait that nothing completes returns an error status
    (the kernel exits normally; the context stays usable)."""
    bd.bitdelta_set_wait_limit_ns(5_000_000)   # 5 ms
    try:
        bd.bitdelta_debug_wait_timeout()
        assert bd.bitdelta_check_error() == 6   # BD_ERR_DEVICE_TIMEOUT
        assert bd.bitdelta_check_error() == 0   # cleared
    finally:
        bd.bitdelta_set_wait_limit_ns(2_000_000_000)
    # the context still works
    wb, packed, alpha = _layer(0, 64, 128, True)
    x = synth.activations(0, 2, 128)
    assert_linear_close(bf16_values(_run(x, wb, packed, alpha, True)),
                        oracle.linear(x, wb, packed, alpha, True))


@pytest.mark.parametrize("shape", [(37, 256), (250, 1024), (1, 128), (17, 384), (5003, 256)])
@pytest.mark.parametrize("M", [1, 5, 8, 9, 12, 16])
def test_decode_ring_ragged_d_out(shape, M):
    """d_in a multiple of 128 (the cp.async ring for M <= 8, and for M = 9..16
    on grids of one wave; 5003 rows make a grid of more than two CTAs per SM,
    where M > 8 goes to the register kernel) with a d_out that leaves the last
    CTA a partial group of 16 rows, and empty token slots."""
    d_out, d_in = shape
    wb, packed, alpha = _layer(3, d_out, d_in, True)
    x = synth.activations(3, M, d_in)
    y = _run(x, wb, packed, alpha, True)
    assert bd.bitdelta_check_error() == 0
    assert_linear_close(bf16_values(y), oracle.linear(x, wb, packed, alpha, True),
                        f"{shape} M={M}")


@pytest.mark.parametrize("M", [2, 8, 16])
def test_decode_unaligned_sign_rows(M):
    """Packed signs starting 8 bytes past a 16-byte boundary on a d_in that
    the ring could take: the register kernel with byte-wise sign loads runs
    instead, and matches the oracle."""
    import torch
    d_out, d_in = 96, 512
    wb, packed, alpha = _layer(4, d_out, d_in, True)
    raw = torch.empty(packed.size + 8, dtype=torch.uint8, device="cuda")
    shifted = raw[8:8 + packed.size].view(packed.shape)
    shifted.copy_(bd_tensor(packed))
    assert shifted.data_ptr() % 16 == 8
    x = synth.activations(4, M, d_in)
    y = bd.bitdelta_linear(to_dev_bf16(x), to_dev_bf16(wb), shifted, bd_tensor(alpha),
                           per_row=True)
    assert bd.bitdelta_check_error() == 0
    assert_linear_close(bf16_values(y), oracle.linear(x, wb, packed, alpha, True), f"M={M}")
