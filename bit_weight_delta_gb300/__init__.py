"""Thin Python binding of libbitdelta.so (the GB300 BitDelta hot path).

Every function here only marshals arguments: it checks tensor devices and
dtypes, allocates outputs through torch (device memory is plumbing), and calls
the C entry point of the same name declared in include/bitdelta.h.  All
arithmetic runs in the library's CUDA kernels; there is no CPU or PyTorch
fallback.  If the library cannot be loaded, importing works but every call
raises.

bf16 tensors are torch.bfloat16; the packed sign matrix is torch.uint8
[d_out, d_in/8]; alpha is torch.float32 ([1] or [d_out]).
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import _build

PER_MATRIX = 0
PER_ROW = 1

_STATUS = {
    0: "BD_OK", 1: "BD_ERR_INVALID_ARG", 2: "BD_ERR_UNSUPPORTED_SHAPE", 3: "BD_ERR_MISALIGNED",
    4: "BD_ERR_WORKSPACE", 5: "BD_ERR_CUDA", 6: "BD_ERR_DEVICE_TIMEOUT",
    7: "BD_ERR_DEVICE_BOUNDS", 8: "BD_ERR_CACHE_FULL",
}

EXPORTED = (
    "bitdelta_packed_bytes", "bitdelta_compress_workspace_bytes", "bitdelta_compress",
    "bitdelta_reconstruct", "bitdelta_linear", "bitdelta_linear_ws",
    "bitdelta_linear_workspace_bytes", "bitdelta_linear_grouped",
    "bitdelta_check_error", "bitdelta_set_wait_limit_ns", "bitdelta_debug_wait_timeout",
    "bitdelta_debug_split_schedule",
    "bitdelta_set_prefill_tile",
    "bitdelta_status_string", "bitdelta_compress_noalloc", "bitdelta_sign_similarity",
    "bitdelta_sign_similarity_workspace_bytes", "bitdelta_monosoup",
    "bitdelta_monosoup_workspace_bytes",
)
CACHE_EXPORTED = (
    "bd_cache_create", "bd_cache_destroy", "bd_cache_register", "bd_cache_acquire",
    "bd_cache_release", "bd_cache_get_stats", "bd_cache_slot_of",
)
KMERGE_EXPORTED = (
    "bd_kmerge_create", "bd_kmerge_destroy", "bd_kmerge_request", "bd_kmerge_commit",
    "bd_kmerge_entry_of", "bd_kmerge_entry_info", "bd_kmerge_get_stats",
)


class BitDeltaError(RuntimeError):
    def __init__(self, fn: str, code: int):
        self.code = code
        super().__init__(f"{fn} failed: {_STATUS.get(code, code)} ({status_string(code)})")


_lib = None


def library_path() -> str:
    return _build.LIB_PATH


def load(build_if_missing: bool = True) -> ctypes.CDLL:
    """Load libbitdelta.so (building it in-tree first if it is missing or stale)."""
    global _lib
    if _lib is not None:
        return _lib
    if build_if_missing:
        _build.build()
    if not os.path.exists(_build.LIB_PATH):
        raise RuntimeError(f"libbitdelta.so not found at {_build.LIB_PATH}; run the build")
    lib = ctypes.CDLL(_build.LIB_PATH)
    i64, i32, p, sz = ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p, ctypes.c_size_t
    st = ctypes.c_int
    lib.bitdelta_packed_bytes.argtypes = [i64, i64]
    lib.bitdelta_packed_bytes.restype = sz
    lib.bitdelta_compress_workspace_bytes.argtypes = [i64, i64, st]
    lib.bitdelta_compress_workspace_bytes.restype = sz
    lib.bitdelta_compress.argtypes = [p, p, i64, i64, st, p, p, p, sz, p]
    lib.bitdelta_compress.restype = st
    lib.bitdelta_compress_noalloc.argtypes = [p, p, i64, i64, st, p, p, p]
    lib.bitdelta_compress_noalloc.restype = st
    lib.bitdelta_reconstruct.argtypes = [p, p, p, st, i64, i64, p, p]
    lib.bitdelta_reconstruct.restype = st
    lib.bitdelta_linear.argtypes = [p, i64, p, p, p, st, i64, i64, p, p]
    lib.bitdelta_linear.restype = st
    lib.bitdelta_linear_ws.argtypes = [p, i64, p, p, p, st, i64, i64, p, p, sz, p]
    lib.bitdelta_linear_ws.restype = st
    lib.bitdelta_linear_workspace_bytes.argtypes = [i64, i64, i64]
    lib.bitdelta_linear_workspace_bytes.restype = sz
    lib.bitdelta_linear_grouped.argtypes = [p, i64, p, p, i32, i32, p, p, p, i32, st, i64, i64,
                                            p, p]
    lib.bitdelta_linear_grouped.restype = st
    lib.bitdelta_check_error.argtypes = [p]
    lib.bitdelta_check_error.restype = st
    lib.bitdelta_set_wait_limit_ns.argtypes = [ctypes.c_uint64]
    lib.bitdelta_set_wait_limit_ns.restype = st
    lib.bitdelta_set_prefill_tile.argtypes = [ctypes.c_int]
    lib.bitdelta_set_prefill_tile.restype = st
    lib.bitdelta_debug_wait_timeout.argtypes = [p]
    lib.bitdelta_debug_wait_timeout.restype = st
    lib.bitdelta_debug_split_schedule.argtypes = [i64, i64, i64, i64, i64, p, i64,
                                                  ctypes.POINTER(i64)]
    lib.bitdelta_debug_split_schedule.restype = st
    lib.bitdelta_status_string.argtypes = [st]
    lib.bitdelta_status_string.restype = ctypes.c_char_p
    lib.bitdelta_sign_similarity_workspace_bytes.argtypes = [i64, i32]
    lib.bitdelta_sign_similarity_workspace_bytes.restype = sz
    lib.bitdelta_sign_similarity.argtypes = [p, p, p, p, i32, st, i64, i64, p, p, p, sz, p]
    lib.bitdelta_sign_similarity.restype = st
    lib.bitdelta_monosoup_workspace_bytes.argtypes = [i64, i64, i32, i32]
    lib.bitdelta_monosoup_workspace_bytes.restype = sz
    lib.bitdelta_monosoup.argtypes = [p, p, i32, i32, i32, ctypes.c_uint64, i64, i64, p, p, p,
                                      sz, p]
    lib.bitdelta_monosoup.restype = st
    lib.bd_cache_create.argtypes = [p, sz, sz, i32, st, p, ctypes.POINTER(p)]
    lib.bd_cache_destroy.argtypes = [p]
    lib.bd_cache_register.argtypes = [p, i32, p, sz]
    lib.bd_cache_acquire.argtypes = [p, i32, p, ctypes.POINTER(p)]
    lib.bd_cache_release.argtypes = [p, i32, p]
    lib.bd_cache_get_stats.argtypes = [p, ctypes.POINTER(_CacheStats)]
    lib.bd_cache_slot_of.argtypes = [p, i32, ctypes.POINTER(i32)]
    for name in CACHE_EXPORTED:
        getattr(lib, name).restype = st
    u64 = ctypes.c_uint64
    lib.bd_kmerge_create.argtypes = [u64, ctypes.POINTER(p)]
    lib.bd_kmerge_destroy.argtypes = [p]
    lib.bd_kmerge_request.argtypes = [p, i32, u64, p, i32, ctypes.POINTER(ctypes.c_int),
                                      ctypes.POINTER(i32)]
    lib.bd_kmerge_commit.argtypes = [p, i32, i32, i32, u64]
    lib.bd_kmerge_entry_of.argtypes = [p, i32, ctypes.POINTER(i32)]
    lib.bd_kmerge_entry_info.argtypes = [p, i32, ctypes.POINTER(u64), ctypes.POINTER(i32)]
    lib.bd_kmerge_get_stats.argtypes = [p, ctypes.POINTER(_KMergeStats)]
    for name in KMERGE_EXPORTED:
        getattr(lib, name).restype = st
    _lib = lib
    return lib


def status_string(code: int) -> str:
    return load().bitdelta_status_string(int(code)).decode()


def _check(fn: str, code: int) -> None:
    if code != 0:
        raise BitDeltaError(fn, code)


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _ptr(t: torch.Tensor | None) -> ctypes.c_void_p:
    return ctypes.c_void_p(0 if t is None else t.data_ptr())


def _dev(t: torch.Tensor, dtype, name: str) -> torch.Tensor:
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def _mode(per_row: bool) -> int:
    return PER_ROW if per_row else PER_MATRIX


def bitdelta_packed_bytes(d_out: int, d_in: int) -> int:
    return int(load().bitdelta_packed_bytes(d_out, d_in))


def bitdelta_compress_workspace_bytes(d_out: int, d_in: int, per_row: bool) -> int:
    return int(load().bitdelta_compress_workspace_bytes(d_out, d_in, _mode(per_row)))


def bitdelta_compress(w_base, w_ft, per_row: bool = True, packed_out=None, alpha_out=None,
                      workspace=None, stream=None):
    """Packed signs and α of Δ = W_ft − W_base.  Returns (packed, alpha)."""
    _dev(w_base, torch.bfloat16, "w_base")
    _dev(w_ft, torch.bfloat16, "w_ft")
    d_out, d_in = w_base.shape
    if packed_out is None:
        packed_out = torch.empty((d_out, d_in // 8), dtype=torch.uint8, device=w_base.device)
    if alpha_out is None:
        alpha_out = torch.empty((d_out if per_row else 1,), dtype=torch.float32,
                                device=w_base.device)
    need = bitdelta_compress_workspace_bytes(d_out, d_in, per_row)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=w_base.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("bitdelta_compress", load().bitdelta_compress(
        _ptr(w_base), _ptr(w_ft), d_out, d_in, _mode(per_row), _ptr(packed_out), _ptr(alpha_out),
        _ptr(workspace), ws_bytes, _stream(stream)))
    return packed_out, alpha_out


def bitdelta_compress_noalloc(w_base, w_ft, per_row: bool, packed_out, alpha_out, stream=None):
    """bitdelta_compress for callers that cannot allocate device memory: the
    outputs are passed in and the library allocates nothing (per-matrix α
    uses a fixed device array, d_out <= 65536).  Returns (packed, alpha)."""
    _dev(w_base, torch.bfloat16, "w_base")
    _dev(w_ft, torch.bfloat16, "w_ft")
    _dev(packed_out, torch.uint8, "packed_out")
    _dev(alpha_out, torch.float32, "alpha_out")
    d_out, d_in = w_base.shape
    _check("bitdelta_compress_noalloc", load().bitdelta_compress_noalloc(
        _ptr(w_base), _ptr(w_ft), d_out, d_in, _mode(per_row), _ptr(packed_out),
        _ptr(alpha_out), _stream(stream)))
    return packed_out, alpha_out


def bitdelta_reconstruct(w_base, packed, alpha, per_row: bool = True, out=None, stream=None):
    """W_eff = bf16(fp32(W_base) ± α) written to memory."""
    _dev(w_base, torch.bfloat16, "w_base")
    _dev(packed, torch.uint8, "packed")
    _dev(alpha, torch.float32, "alpha")
    d_out, d_in = w_base.shape
    if out is None:
        out = torch.empty_like(w_base)
    _check("bitdelta_reconstruct", load().bitdelta_reconstruct(
        _ptr(w_base), _ptr(packed), _ptr(alpha), _mode(per_row), d_out, d_in, _ptr(out),
        _stream(stream)))
    return out


def bitdelta_linear(x, w_base, packed, alpha, per_row: bool = True, out=None, stream=None):
    """y = x · (W_base + α·sign(Δ))ᵀ, x [..., d_in] bf16 -> y [..., d_out] bf16."""
    _dev(x, torch.bfloat16, "x")
    _dev(w_base, torch.bfloat16, "w_base")
    _dev(packed, torch.uint8, "packed")
    _dev(alpha, torch.float32, "alpha")
    d_out, d_in = w_base.shape
    lead = x.shape[:-1]
    M = x.numel() // d_in if x.numel() else 0
    if out is None:
        out = torch.empty((*lead, d_out), dtype=torch.bfloat16, device=x.device)
    _check("bitdelta_linear", load().bitdelta_linear(
        _ptr(x), M, _ptr(w_base), _ptr(packed), _ptr(alpha), _mode(per_row), d_out, d_in,
        _ptr(out), _stream(stream)))
    return out


def bitdelta_linear_workspace_bytes(M: int, d_out: int, d_in: int) -> int:
    """Bytes of the split-schedule workspace of bitdelta_linear_ws (0: never split)."""
    return int(load().bitdelta_linear_workspace_bytes(M, d_out, d_in))


def bitdelta_linear_ws(x, w_base, packed, alpha, workspace, per_row: bool = True, out=None,
                       stream=None):
    """bitdelta_linear with a split-schedule workspace (uint8 CUDA tensor on a
    256-byte boundary of at least bitdelta_linear_workspace_bytes(M, d_out,
    d_in) bytes, or None)."""
    _dev(x, torch.bfloat16, "x")
    _dev(w_base, torch.bfloat16, "w_base")
    _dev(packed, torch.uint8, "packed")
    _dev(alpha, torch.float32, "alpha")
    d_out, d_in = w_base.shape
    lead = x.shape[:-1]
    M = x.numel() // d_in if x.numel() else 0
    if out is None:
        out = torch.empty((*lead, d_out), dtype=torch.bfloat16, device=x.device)
    ws_bytes = 0
    if workspace is not None:
        _dev(workspace, torch.uint8, "workspace")
        ws_bytes = workspace.numel()
    _check("bitdelta_linear_ws", load().bitdelta_linear_ws(
        _ptr(x), M, _ptr(w_base), _ptr(packed), _ptr(alpha), _mode(per_row), d_out, d_in,
        _ptr(out), _ptr(workspace), ws_bytes, _stream(stream)))
    return out


def variant_tables(packed_list, alpha_list, device):
    """Device arrays of the variants' packed and α pointers (slot v-1 = variant v).

    The returned tensors must stay alive while the tables are used; the
    caller keeps them together with the listed tensors."""
    pk = torch.tensor([t.data_ptr() for t in packed_list] or [0], dtype=torch.int64,
                      device=device)
    al = torch.tensor([t.data_ptr() for t in alpha_list] or [0], dtype=torch.int64,
                      device=device)
    return pk, al


def bitdelta_linear_grouped(x, seg_offsets, seg_variant, w_base, packed_table, alpha_table,
                            n_var: int, max_seg_len: int, per_row: bool = True, out=None,
                            stream=None):
    """Multi-tenant linear: rows of segment s use variant seg_variant[s] (0 = base).

    seg_offsets int32 [n_seg+1] and seg_variant int32 [n_seg] are CUDA tensors;
    packed_table / alpha_table are int64 CUDA tensors of device pointers, as
    made by variant_tables()."""
    _dev(x, torch.bfloat16, "x")
    _dev(w_base, torch.bfloat16, "w_base")
    _dev(seg_offsets, torch.int32, "seg_offsets")
    _dev(seg_variant, torch.int32, "seg_variant")
    d_out, d_in = w_base.shape
    M = x.shape[0]
    if out is None:
        out = torch.empty((M, d_out), dtype=torch.bfloat16, device=x.device)
    _check("bitdelta_linear_grouped", load().bitdelta_linear_grouped(
        _ptr(x), M, _ptr(seg_offsets), _ptr(seg_variant), seg_variant.numel(), int(max_seg_len),
        _ptr(w_base), _ptr(packed_table), _ptr(alpha_table), int(n_var), _mode(per_row), d_out,
        d_in, _ptr(out), _stream(stream)))
    return out


def bitdelta_check_error(stream=None) -> int:
    """Synchronise and return (then clear) the device error status code."""
    return int(load().bitdelta_check_error(_stream(stream)))


def bitdelta_set_wait_limit_ns(ns: int) -> None:
    _check("bitdelta_set_wait_limit_ns", load().bitdelta_set_wait_limit_ns(int(ns)))


PREFILL_TILES = {"auto": 0, 256: 1, 512: 2}


def bitdelta_set_prefill_tile(tile="auto") -> None:
    """Token width of the tensor-core kernel's pair tiles: "auto", 256 or 512."""
    if tile not in PREFILL_TILES:
        raise ValueError(f"prefill tile must be one of {list(PREFILL_TILES)}, not {tile!r}")
    _check("bitdelta_set_prefill_tile", load().bitdelta_set_prefill_tile(PREFILL_TILES[tile]))


def bitdelta_debug_wait_timeout(stream=None) -> None:
    _check("bitdelta_debug_wait_timeout", load().bitdelta_debug_wait_timeout(_stream(stream)))


def bitdelta_sign_similarity(packed_a, alpha_a, packed_table, alpha_table, n_b: int,
                             per_row: bool = True, out=None, best=None, workspace=None,
                             stream=None):
    """Cosines of the candidate's 1-bit task vector with n_b pool members (page
    section K-Merge).  packed_table / alpha_table: int64 CUDA tensors of device
    pointers (variant_tables()).  Returns (cos [n_b] float64, best [1] int32),
    both CUDA tensors; out / best / workspace (uint8, at least
    bitdelta_sign_similarity_workspace_bytes() + 256 bytes) may be passed in
    to avoid allocations."""
    _dev(packed_a, torch.uint8, "packed_a")
    _dev(alpha_a, torch.float32, "alpha_a")
    d_out, row_bytes = packed_a.shape
    need = bitdelta_sign_similarity_workspace_bytes(d_out, n_b)
    if workspace is None:
        workspace = torch.empty(need + 256, dtype=torch.uint8, device=packed_a.device)
    off = (-workspace.data_ptr()) % 256
    if out is None:
        out = torch.empty(n_b, dtype=torch.float64, device=packed_a.device)
    if best is None:
        best = torch.empty(1, dtype=torch.int32, device=packed_a.device)
    _check("bitdelta_sign_similarity", load().bitdelta_sign_similarity(
        _ptr(packed_a), _ptr(alpha_a), _ptr(packed_table), _ptr(alpha_table), n_b,
        _mode(per_row), d_out, row_bytes * 8, _ptr(out), _ptr(best),
        ctypes.c_void_p(workspace.data_ptr() + off), workspace.numel() - off, _stream(stream)))
    return out, best


def bitdelta_sign_similarity_workspace_bytes(d_out: int, n_b: int) -> int:
    return int(load().bitdelta_sign_similarity_workspace_bytes(d_out, n_b))


def bitdelta_monosoup_workspace_bytes(d_out: int, d_in: int, k: int, rank: int) -> int:
    return int(load().bitdelta_monosoup_workspace_bytes(d_out, d_in, k, rank))


def bitdelta_monosoup(w_base, w_fts, rank: int, power_iters: int = 2, seed: int = 0,
                      out=None, correction=None, workspace=None, stream=None):
    """MonoSoup merge (page section MonoSoup): W_base + (1/k)·Σ rank-r truncated
    SVD of each W_i − W_base.  w_fts: list of k bf16 CUDA tensors shaped like
    w_base.  Returns W_merged (bf16); `correction` (float32 CUDA tensor, same
    shape) receives (1/k)·Σ τ_i when given; `workspace` (uint8, at least
    bitdelta_monosoup_workspace_bytes() + 256 bytes) may be passed in."""
    _dev(w_base, torch.bfloat16, "w_base")
    d_out, d_in = w_base.shape
    k = len(w_fts)
    for i, w in enumerate(w_fts):
        _dev(w, torch.bfloat16, f"w_fts[{i}]")
        if tuple(w.shape) != (d_out, d_in):
            raise ValueError("every checkpoint must have the shape of w_base")
    if out is None:
        out = torch.empty_like(w_base)
    if correction is not None:
        _dev(correction, torch.float32, "correction")
    need = bitdelta_monosoup_workspace_bytes(d_out, d_in, max(k, 1), rank)
    if workspace is None:
        workspace = torch.empty(need + 256, dtype=torch.uint8, device=w_base.device)
    off = (-workspace.data_ptr()) % 256
    table = (ctypes.c_void_p * max(k, 1))(*[w.data_ptr() for w in w_fts])
    _check("bitdelta_monosoup", load().bitdelta_monosoup(
        _ptr(w_base), ctypes.cast(table, ctypes.c_void_p), k, rank, power_iters, seed, d_out,
        d_in, _ptr(out), _ptr(correction) if correction is not None else None,
        ctypes.c_void_p(workspace.data_ptr() + off), workspace.numel() - off, _stream(stream)))
    return out


# --------------------------------------------------------------------------- delta cache


class _CacheStats(ctypes.Structure):
    _fields_ = [(n, ctypes.c_uint64) for n in
                ("acquires", "hits", "queued_behind_load", "loads", "evictions", "bytes_loaded")]


class DeltaCache:
    """The delta cache of include/bitdelta_cache.h over a caller-owned arena.

    arena: a contiguous uint8 tensor, CUDA (device arena: loads are async
    host-to-device copies on `copy_stream`) or CPU (host arena: loads are
    memcpy, no CUDA).  Variants are registered as contiguous CPU uint8
    tensors (pinned memory lets the copies run asynchronously); the caller
    keeps them alive.  acquire() returns a uint8 view of the variant's bytes
    in the arena, valid until the matching release()."""

    def __init__(self, arena: torch.Tensor, slot_bytes: int, pin_top_k: int = 6,
                 copy_stream=None):
        if arena.dtype != torch.uint8 or not arena.is_contiguous():
            raise ValueError("arena must be a contiguous uint8 tensor")
        self.arena = arena
        self.device = arena.is_cuda
        self.copy_stream = (copy_stream if copy_stream is not None else
                            (torch.cuda.Stream(device=arena.device) if self.device else None))
        handle = ctypes.c_void_p()
        cs = ctypes.c_void_p(self.copy_stream.cuda_stream if self.device else 0)
        _check("bd_cache_create", load().bd_cache_create(
            _ptr(arena), arena.numel(), slot_bytes, pin_top_k, 0 if self.device else 1, cs,
            ctypes.byref(handle)))
        self.handle = handle
        self.slot_bytes = slot_bytes
        self._blobs = {}

    def register(self, variant: int, blob: torch.Tensor) -> None:
        if blob.is_cuda or blob.dtype != torch.uint8 or not blob.is_contiguous():
            raise ValueError("a variant's blob must be a contiguous CPU uint8 tensor")
        _check("bd_cache_register", load().bd_cache_register(self.handle, variant, _ptr(blob),
                                                             blob.numel()))
        self._blobs[variant] = blob

    def _s(self, stream) -> ctypes.c_void_p:
        return _stream(stream) if self.device else ctypes.c_void_p(0)

    def acquire(self, variant: int, stream=None) -> torch.Tensor:
        ptr = ctypes.c_void_p()
        _check("bd_cache_acquire", load().bd_cache_acquire(self.handle, variant, self._s(stream),
                                                           ctypes.byref(ptr)))
        off = ptr.value - self.arena.data_ptr()
        return self.arena[off:off + self._blobs[variant].numel()]

    def release(self, variant: int, stream=None) -> None:
        _check("bd_cache_release", load().bd_cache_release(self.handle, variant,
                                                           self._s(stream)))

    def try_acquire(self, variant: int, stream=None):
        """acquire(), or None when the cache is full (BD_ERR_CACHE_FULL)."""
        try:
            return self.acquire(variant, stream)
        except BitDeltaError as e:
            if e.code == 8:
                return None
            raise

    def slot_of(self, variant: int) -> int:
        slot = ctypes.c_int32()
        _check("bd_cache_slot_of", load().bd_cache_slot_of(self.handle, variant,
                                                           ctypes.byref(slot)))
        return slot.value

    def stats(self) -> dict:
        st = _CacheStats()
        _check("bd_cache_get_stats", load().bd_cache_get_stats(self.handle, ctypes.byref(st)))
        return {n: int(getattr(st, n)) for n, _ in _CacheStats._fields_}

    def close(self) -> None:
        if self.handle is not None:
            _check("bd_cache_destroy", load().bd_cache_destroy(self.handle))
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


# --------------------------------------------------------------------------- K-Merge pool


class _KMergeStats(ctypes.Structure):
    _fields_ = [("entries", ctypes.c_int32), ("adapters", ctypes.c_int32)] + [
        (n, ctypes.c_uint64) for n in ("used_bytes", "budget_bytes", "stores", "merges_proposed",
                                       "merges_accepted", "merges_rejected", "rejects", "hits")]


class KMergePool:
    """The K-Merge adapter pool of include/bitdelta_kmerge.h (host policy).

    request(adapter, nbytes, cos=None) returns (action, entry), action one of
    "hit", "store", "need_similarity", "merge", "reject"; after "merge" the
    caller merges the adapter into the entry and reports the outcome with
    commit().  Similarities come from bitdelta_sign_similarity against the
    entries' stored deltas (see request_on_device)."""

    ACTIONS = ("hit", "store", "need_similarity", "merge", "reject")

    def __init__(self, budget_bytes: int):
        handle = ctypes.c_void_p()
        _check("bd_kmerge_create", load().bd_kmerge_create(budget_bytes, ctypes.byref(handle)))
        self.handle = handle

    def request(self, adapter: int, nbytes: int, cos=None):
        action, entry = ctypes.c_int(), ctypes.c_int32()
        if cos is None:
            cptr, n = None, 0
            keep = None
        else:
            keep = (ctypes.c_double * max(len(cos), 1))(*[float(c) for c in cos])
            cptr, n = ctypes.cast(keep, ctypes.c_void_p), len(cos)
        _check("bd_kmerge_request", load().bd_kmerge_request(
            self.handle, adapter, nbytes, cptr, n, ctypes.byref(action), ctypes.byref(entry)))
        return self.ACTIONS[action.value], entry.value

    def request_on_device(self, adapter: int, nbytes: int, packed, alpha, entry_packed,
                          entry_alpha, per_row: bool = True):
        """request(); when the pool needs the similarities, computes them on
        the GPU (bitdelta_sign_similarity of the adapter's packed/alpha with
        every entry's, in entry order) and requests again.  Returns (action,
        entry, cos) with cos a CPU float64 tensor or None."""
        action, entry = self.request(adapter, nbytes)
        if action != "need_similarity":
            return action, entry, None
        parts = []
        for lo in range(0, len(entry_packed), 256):   # at most 256 members per call
            ep, ea = list(entry_packed[lo:lo + 256]), list(entry_alpha[lo:lo + 256])
            pt, at = variant_tables(ep, ea, packed.device)
            cos, _ = bitdelta_sign_similarity(packed, alpha, pt, at, len(ep), per_row)
            parts.append(cos.cpu())
        cos_h = torch.cat(parts)
        action, entry = self.request(adapter, nbytes, cos_h.tolist())
        return action, entry, cos_h

    def commit(self, adapter: int, entry: int, accepted: bool, merged_bytes: int) -> None:
        _check("bd_kmerge_commit", load().bd_kmerge_commit(self.handle, adapter, entry,
                                                           1 if accepted else 0, merged_bytes))

    def entry_of(self, adapter: int) -> int:
        e = ctypes.c_int32()
        _check("bd_kmerge_entry_of", load().bd_kmerge_entry_of(self.handle, adapter,
                                                               ctypes.byref(e)))
        return e.value

    def entry_info(self, entry: int):
        b, n = ctypes.c_uint64(), ctypes.c_int32()
        _check("bd_kmerge_entry_info", load().bd_kmerge_entry_info(
            self.handle, entry, ctypes.byref(b), ctypes.byref(n)))
        return int(b.value), int(n.value)

    def stats(self) -> dict:
        st = _KMergeStats()
        _check("bd_kmerge_get_stats", load().bd_kmerge_get_stats(self.handle, ctypes.byref(st)))
        return {n: int(getattr(st, n)) for n, _ in _KMergeStats._fields_}

    def close(self) -> None:
        if self.handle is not None:
            _check("bd_kmerge_destroy", load().bd_kmerge_destroy(self.handle))
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
