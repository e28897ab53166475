"""bitdelta_compress_noalloc: compression for callers that cannot allocate
device memory (e.g. a plug-in handed finished buffers by its host framework,
or a serving loop whose device memory is planned up front), through the C ABI.

Its output must match bitdelta_compress, the entry point that takes a caller
workspace: packed signs bit for bit, α within 1e-6 relative, on two calls in a
row (the second call reuses the library's fixed scratch array, which must not
carry the first call's state into the result).  At the scratch array's row
limit it is also checked against the oracle directly.  This file is
collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

import bit_weight_delta_gb300 as bd
import oracle
import synth.device as sd
from gpu_util import from_dev_bf16

pytestmark = pytest.mark.gpu

ALPHA_RTOL = 1e-6


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def _noalloc(lib, wb, wf, per_row, packed, alpha):
    d_out, d_in = wb.shape
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.bitdelta_compress_noalloc(_p(wb), _p(wf), d_out, d_in, 1 if per_row else 0,
                                         _p(packed), _p(alpha), stream)


@pytest.mark.parametrize("per_row", [False, True])
@pytest.mark.parametrize("shape", [(4096, 4096), (300, 1032), (65536, 256)])
def test_noalloc_matches_workspace_entry_point(shape, per_row):
    lib = bd.load()
    torch.cuda.set_device(0)
    d_out, d_in = shape
    for call in range(2):   # two calls in a row through the shared scratch
        wb, wf = sd.layer(40 + call, d_out, d_in, stream=call)
        ref_packed, ref_alpha = bd.bitdelta_compress(wb, wf, per_row=per_row)
        packed = torch.full((d_out, d_in // 8), 0xA5, dtype=torch.uint8, device="cuda")
        alpha = torch.full((d_out if per_row else 1,), -1.0, dtype=torch.float32, device="cuda")
        assert _noalloc(lib, wb, wf, per_row, packed, alpha) == 0
        assert bd.bitdelta_check_error() == 0
        assert torch.equal(packed, ref_packed), f"call {call}: packed signs differ"
        a = alpha.double().cpu().numpy()
        r = ref_alpha.double().cpu().numpy()
        assert np.all(np.abs(a - r) <= ALPHA_RTOL * np.abs(r)), f"call {call}: alpha differs"


def test_noalloc_rejects_rows_beyond_the_scratch():
    """Per-matrix α needs 8 bytes of scratch per row: more than 65536 rows is
    refused with BD_ERR_WORKSPACE before anything is launched."""
    lib = bd.load()
    wb = torch.empty((65537, 8), dtype=torch.bfloat16, device="cuda")
    packed = torch.empty((65537, 1), dtype=torch.uint8, device="cuda")
    alpha = torch.empty((1,), dtype=torch.float32, device="cuda")
    assert _noalloc(lib, wb, wb, False, packed, alpha) == 4   # BD_ERR_WORKSPACE


def test_noalloc_at_the_row_limit_matches_the_oracle():
    """65536 rows, per-matrix α (the largest problem the scratch array takes),
    two calls in a row on different inputs: signs bit for bit and α within
    1e-6 of the oracle's fp64 mean |Δ| ("Mathematical foundation")."""
    lib = bd.load()
    torch.cuda.set_device(0)
    d_out, d_in = 65536, 256
    for call in range(2):
        wb, wf = sd.layer(50 + call, d_out, d_in, stream=call)
        packed = torch.full((d_out, d_in // 8), 0x5A, dtype=torch.uint8, device="cuda")
        alpha = torch.full((1,), -1.0, dtype=torch.float32, device="cuda")
        assert _noalloc(lib, wb, wf, False, packed, alpha) == 0
        assert bd.bitdelta_check_error() == 0
        p_ref, _, a64 = oracle.compress(from_dev_bf16(wb), from_dev_bf16(wf), False)
        assert np.array_equal(packed.cpu().numpy(), p_ref), f"call {call}: packed signs differ"
        a = float(alpha.double().item())
        assert abs(a - a64[0]) <= ALPHA_RTOL * abs(a64[0]), f"call {call}: alpha {a} vs {a64[0]}"
