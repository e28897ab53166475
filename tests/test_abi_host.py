"""The C ABI library loads, exports every declared symbol, and rejects bad
arguments on the host before touching the GPU (no GPU needed: every call here
returns before any CUDA API call)."""
import ctypes
import os
import re
import subprocess

import pytest

import bit_weight_delta_gb300 as bd

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "bitdelta.h")

OK, INVALID, SHAPE, MISALIGNED, WORKSPACE = 0, 1, 2, 3, 4
BAD = ctypes.c_void_p(0x1001)     # never dereferenced: rejected as misaligned first
GOOD = ctypes.c_void_p(0x100000)  # 16-byte aligned fake address, never dereferenced
NULL = ctypes.c_void_p(0)


@pytest.fixture(scope="module")
def lib():
    return bd.load()


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"\b(bitdelta_\w+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for required in ("bitdelta_compress", "bitdelta_reconstruct", "bitdelta_linear",
                     "bitdelta_linear_grouped", "bitdelta_check_error"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", bd.library_path()], capture_output=True,
                         text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    for name in declared_functions():
        assert name in exported, name
        assert hasattr(lib, name)
    assert set(bd.EXPORTED) == set(declared_functions())


def test_library_exports_the_delta_cache(lib):
    text = open(os.path.join(os.path.dirname(HEADER), "bitdelta_cache.h")).read()
    declared = sorted(set(re.findall(r"\b(bd_cache_\w+)\s*\(", text)))
    out = subprocess.run(["nm", "-D", "--defined-only", bd.library_path()], capture_output=True,
                         text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    assert declared and set(declared) <= exported
    assert set(bd.CACHE_EXPORTED) == set(declared)


def test_library_exports_the_kmerge_pool(lib):
    text = open(os.path.join(os.path.dirname(HEADER), "bitdelta_kmerge.h")).read()
    declared = sorted(set(re.findall(r"\b(bd_kmerge_\w+)\s*\(", text)))
    out = subprocess.run(["nm", "-D", "--defined-only", bd.library_path()], capture_output=True,
                         text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    assert declared and set(declared) <= exported
    assert set(bd.KMERGE_EXPORTED) == set(declared)


def test_packed_bytes_and_workspace(lib):
    assert bd.bitdelta_packed_bytes(4096, 4096) == 4096 * 512   # "Infrastructure details"
    assert bd.bitdelta_packed_bytes(8, 16) == 16
    assert bd.bitdelta_packed_bytes(8, 12) == 0                  # d_in % 8 != 0
    assert bd.bitdelta_compress_workspace_bytes(4096, 4096, per_row=True) == 0
    assert bd.bitdelta_compress_workspace_bytes(4096, 4096, per_row=False) == 8 * 4096 + 256


def test_status_strings(lib):
    for code in range(9):
        assert bd.status_string(code) != "unknown status"
    assert bd.status_string(99) == "unknown status"


def test_compress_rejects_bad_arguments(lib):
    f = lib.bitdelta_compress
    assert f(NULL, GOOD, 8, 16, 1, GOOD, GOOD, NULL, 0, NULL) == INVALID
    assert f(GOOD, GOOD, 8, 16, 7, GOOD, GOOD, NULL, 0, NULL) == INVALID     # bad mode
    assert f(GOOD, GOOD, 0, 16, 1, GOOD, GOOD, NULL, 0, NULL) == INVALID     # d_out 0
    assert f(GOOD, GOOD, 8, 12, 1, GOOD, GOOD, NULL, 0, NULL) == SHAPE       # d_in % 8
    assert f(BAD, GOOD, 8, 16, 1, GOOD, GOOD, NULL, 0, NULL) == MISALIGNED
    assert f(GOOD, GOOD, 8, 16, 0, GOOD, GOOD, NULL, 0, NULL) == WORKSPACE   # per-matrix
    assert f(GOOD, GOOD, 8, 16, 0, GOOD, GOOD, GOOD, 16, NULL) == WORKSPACE  # too small


def test_reconstruct_rejects_bad_arguments(lib):
    f = lib.bitdelta_reconstruct
    assert f(GOOD, NULL, GOOD, 1, 8, 16, GOOD, NULL) == INVALID
    assert f(GOOD, GOOD, GOOD, 1, 8, 20, GOOD, NULL) == SHAPE
    assert f(GOOD, GOOD, GOOD, 1, 8, 16, BAD, NULL) == MISALIGNED


def test_linear_rejects_bad_arguments(lib):
    f = lib.bitdelta_linear
    assert f(GOOD, -1, GOOD, GOOD, GOOD, 1, 8, 16, GOOD, NULL) == INVALID
    assert f(NULL, 4, GOOD, GOOD, GOOD, 1, 8, 16, GOOD, NULL) == INVALID
    assert f(GOOD, 4, GOOD, GOOD, GOOD, 1, 8, 9, GOOD, NULL) == SHAPE
    assert f(BAD, 4, GOOD, GOOD, GOOD, 1, 8, 16, GOOD, NULL) == MISALIGNED
    # M == 0 is a no-op that needs no pointers and no device
    assert f(NULL, 0, NULL, NULL, NULL, 1, 8, 16, NULL, NULL) == OK


def test_grouped_rejects_bad_arguments(lib):
    f = lib.bitdelta_linear_grouped
    args = dict(x=GOOD, M=4, so=GOOD, sv=GOOD, n_seg=1, max_len=4, wb=GOOD, pt=GOOD, at=GOOD,
                n_var=1, mode=1, d_out=8, d_in=16, y=GOOD)

    def call(**kw):
        a = {**args, **kw}
        return f(a["x"], a["M"], a["so"], a["sv"], a["n_seg"], a["max_len"], a["wb"], a["pt"],
                 a["at"], a["n_var"], a["mode"], a["d_out"], a["d_in"], a["y"], NULL)

    assert call(n_seg=-1) == INVALID
    assert call(n_var=-1) == INVALID
    assert call(mode=3) == INVALID
    assert call(so=NULL) == INVALID
    assert call(pt=NULL) == INVALID
    assert call(d_in=10) == SHAPE
    assert call(y=BAD) == MISALIGNED
    assert call(M=0, x=NULL, so=NULL) == OK      # empty batch is a no-op
    assert call(n_seg=0, so=NULL) == OK


def test_monosoup_rejects_bad_arguments(lib):
    f = lib.bitdelta_monosoup
    table = (ctypes.c_void_p * 2)(GOOD.value, GOOD.value)
    ws_need = lib.bitdelta_monosoup_workspace_bytes(64, 128, 2, 8)
    assert ws_need > 0
    args = dict(wb=GOOD, wft=ctypes.cast(table, ctypes.c_void_p), k=2, rank=8, q=2, d_out=64,
                d_in=128, out=GOOD, corr=NULL, ws=GOOD, ws_bytes=ws_need)

    def call(**kw):
        a = {**args, **kw}
        return f(a["wb"], a["wft"], a["k"], a["rank"], a["q"], 7, a["d_out"], a["d_in"],
                 a["out"], a["corr"], a["ws"], a["ws_bytes"], NULL)

    assert call(wb=NULL) == INVALID
    assert call(wft=NULL) == INVALID
    assert call(out=NULL) == INVALID
    assert call(d_in=100) == SHAPE           # d_in % 8 != 0
    assert call(k=0) == SHAPE
    assert call(k=65) == SHAPE
    assert call(rank=65) == SHAPE
    assert call(rank=-1) == SHAPE
    assert call(rank=65, d_out=64) == SHAPE
    assert call(d_out=4, rank=8) == SHAPE     # rank above min(d_out, d_in)
    assert call(q=17) == SHAPE
    assert call(out=BAD) == MISALIGNED
    assert call(corr=BAD) == MISALIGNED
    assert call(ws=BAD) == MISALIGNED
    assert call(ws_bytes=ws_need - 1) == WORKSPACE
    bad_table = (ctypes.c_void_p * 2)(GOOD.value, BAD.value)
    assert call(wft=ctypes.cast(bad_table, ctypes.c_void_p)) == MISALIGNED
    null_table = (ctypes.c_void_p * 2)(GOOD.value, 0)
    assert call(wft=ctypes.cast(null_table, ctypes.c_void_p)) == INVALID
    assert lib.bitdelta_monosoup_workspace_bytes(64, 100, 2, 8) == 0   # bad shape: 0


def test_sign_similarity_rejects_bad_arguments(lib):
    f = lib.bitdelta_sign_similarity
    ws_need = lib.bitdelta_sign_similarity_workspace_bytes(64, 3)
    assert ws_need > 0
    args = dict(pa=GOOD, aa=GOOD, pt=GOOD, at=GOOD, n_b=3, mode=1, d_out=64, d_in=128, cos=GOOD,
                best=GOOD, ws=GOOD, ws_bytes=ws_need)

    def call(**kw):
        a = {**args, **kw}
        return f(a["pa"], a["aa"], a["pt"], a["at"], a["n_b"], a["mode"], a["d_out"], a["d_in"],
                 a["cos"], a["best"], a["ws"], a["ws_bytes"], NULL)

    assert call(pa=NULL) == INVALID
    assert call(pt=NULL) == INVALID
    assert call(cos=NULL) == INVALID
    assert call(mode=5) == INVALID
    assert call(d_in=12) == SHAPE
    assert call(n_b=0) == SHAPE
    assert call(n_b=257) == SHAPE
    assert call(cos=BAD) == MISALIGNED
    assert call(ws=BAD) == MISALIGNED
    assert call(ws_bytes=ws_need - 1) == WORKSPACE
    assert lib.bitdelta_sign_similarity_workspace_bytes(64, 0) == 0


def test_prefill_tile_setting(lib):
    """The pair-tile width setting is host state: the three named values are
    accepted, anything else rejected; the binding maps 'auto', 256, 512."""
    for v in (1, 2, 0):
        assert lib.bitdelta_set_prefill_tile(v) == OK
    for v in (3, -1, 512):
        assert lib.bitdelta_set_prefill_tile(v) == INVALID
    with pytest.raises(ValueError):
        bd.bitdelta_set_prefill_tile(128)
    bd.bitdelta_set_prefill_tile(512)
    bd.bitdelta_set_prefill_tile("auto")


def test_linear_ws_rejects_bad_arguments(lib):
    f = lib.bitdelta_linear_ws
    ws = ctypes.c_void_p(0x200000)     # 256-byte aligned fake address, never dereferenced
    ws_bad = ctypes.c_void_p(0x200010)
    assert f(GOOD, -1, GOOD, GOOD, GOOD, 1, 8, 16, GOOD, ws, 1 << 20, NULL) == INVALID
    assert f(GOOD, 4, GOOD, GOOD, GOOD, 3, 8, 16, GOOD, ws, 1 << 20, NULL) == INVALID
    assert f(GOOD, 4, GOOD, GOOD, GOOD, 1, 8, 16, GOOD, ws_bad, 1 << 20, NULL) == MISALIGNED
    assert f(NULL, 4, GOOD, GOOD, GOOD, 1, 8, 16, GOOD, ws, 1 << 20, NULL) == INVALID
    assert f(GOOD, 4, GOOD, GOOD, GOOD, 1, 8, 9, GOOD, ws, 1 << 20, NULL) == SHAPE
    assert f(NULL, 0, NULL, NULL, NULL, 1, 8, 16, NULL, NULL, 0, NULL) == OK


def test_linear_workspace_bytes_without_split(lib):
    # decode-size calls and shapes the tensor-core kernel does not take never split
    assert lib.bitdelta_linear_workspace_bytes(16, 4096, 4096) == 0
    assert lib.bitdelta_linear_workspace_bytes(2048, 4096, 4104) == 0
    assert lib.bitdelta_linear_workspace_bytes(2048, 4096, 9) == 0
