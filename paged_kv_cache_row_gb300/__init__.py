"""Paged KV-pool attention for GB300 (sm_103a): Python binding of libminisgl.so.

The C library (include/minisgl.h) does all the work in hand-written CUDA
kernels; this module only marshals torch tensors into pointers, sizes and the
current CUDA stream.  There is no fallback: if the library is not built, or a
call fails, an exception is raised.

Entry points (same names as the C ABI):
    minisgl_store_kv(pool, layer, k, v, out_loc)
    minisgl_decode_attn(pool, layer, q, page_table, seq_lens, sm_scale, ...)
    minisgl_extend_attn(pool, layer, q, page_table, cached_lens, extend_lens, q_offsets, sm_scale, ...)
    minisgl_rope_store_kv(pool, layer, q, k, v, positions, cos_sin_cache, out_loc)
    minisgl_check_indices(page_table, lens, num_rows, out_loc)   (debugging aid)
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

from .build import LIB_PATH

__all__ = [
    "KVPool", "minisgl_store_kv", "minisgl_decode_attn", "minisgl_extend_attn",
    "minisgl_decode_workspace_bytes", "minisgl_device_sm_count", "minisgl_debug_timeout_count",
    "kv_pool_bytes", "load_library", "MinisglError", "EXPORTED_SYMBOLS",
    "minisgl_decode_attn_noalloc", "minisgl_rope_store_kv", "minisgl_cascade_decode_attn",
    "minisgl_cascade_workspace_bytes", "minisgl_store_decode_attn", "minisgl_check_indices",
    "minisgl_debug_set_pdl", "extend_work_counter", "minisgl_cascade_extend_attn",
    "minisgl_cascade_extend_workspace_bytes", "minisgl_check_shared_prefix",
]

EXPORTED_SYMBOLS = [
    "minisgl_store_kv", "minisgl_decode_workspace_bytes", "minisgl_decode_attn",
    "minisgl_extend_attn", "minisgl_last_error", "minisgl_device_sm_count",
    "minisgl_debug_timeout_count", "minisgl_decode_attn_noalloc", "minisgl_rope_store_kv",
    "minisgl_cascade_decode_attn", "minisgl_cascade_workspace_bytes", "minisgl_store_decode_attn",
    "minisgl_check_indices", "minisgl_debug_set_pdl", "minisgl_cascade_extend_attn",
    "minisgl_cascade_extend_workspace_bytes", "minisgl_check_shared_prefix",
]

MINISGL_BF16 = 1


class MinisglError(RuntimeError):
    pass


class _PoolDesc(ctypes.Structure):
    _fields_ = [
        ("k_base", ctypes.c_void_p), ("v_base", ctypes.c_void_p),
        ("layer_stride", ctypes.c_int64), ("row_stride", ctypes.c_int64),
        ("num_layers", ctypes.c_int32), ("num_rows", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
        ("page_size", ctypes.c_int32), ("dtype", ctypes.c_int32),
    ]


_lib: Optional[ctypes.CDLL] = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libminisgl.so (built by paged_kv_cache_row_gb300.build)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(f"{path} is missing: build it with `python -m paged_kv_cache_row_gb300.build`"
                          " (or __graft_entry__.build())")
    lib = ctypes.CDLL(path)
    vp, i32, i64, f32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
    P = ctypes.POINTER(_PoolDesc)
    lib.minisgl_store_kv.argtypes = [P, i32, vp, vp, i64, i64, vp, i32, vp]
    lib.minisgl_store_kv.restype = ctypes.c_int
    lib.minisgl_decode_workspace_bytes.argtypes = [i32, i32, i32, i32, i32]
    lib.minisgl_decode_workspace_bytes.restype = sz
    lib.minisgl_decode_attn.argtypes = [P, i32, vp, i32, vp, i32, i64, i32, vp, f32, vp, vp, sz, i32, vp]
    lib.minisgl_decode_attn.restype = ctypes.c_int
    lib.minisgl_decode_attn_noalloc.argtypes = [P, i32, vp, i32, vp, i32, i64, i32, vp, f32, vp, i32, vp]
    lib.minisgl_decode_attn_noalloc.restype = ctypes.c_int
    lib.minisgl_extend_attn.argtypes = [P, i32, vp, i32, vp, i32, i64, i32, vp, vp, vp, i32, f32, vp, vp,
                                        vp]
    lib.minisgl_extend_attn.restype = ctypes.c_int
    lib.minisgl_rope_store_kv.argtypes = [P, i32, vp, i32, i64, vp, vp, i64, i64, vp, vp, i32, vp,
                                          i32, vp]
    lib.minisgl_rope_store_kv.restype = ctypes.c_int
    lib.minisgl_cascade_workspace_bytes.argtypes = [i32, i32, i32, i32]
    lib.minisgl_cascade_workspace_bytes.restype = sz
    lib.minisgl_cascade_decode_attn.argtypes = [P, i32, vp, i32, vp, i32, i64, i32, vp, i32, f32, vp,
                                                vp, sz, vp]
    lib.minisgl_cascade_decode_attn.restype = ctypes.c_int
    lib.minisgl_store_decode_attn.argtypes = [P, i32, vp, vp, i64, i64, vp, vp, i32, vp, i32, i64, i32,
                                              vp, f32, vp, vp, sz, i32, vp]
    lib.minisgl_store_decode_attn.restype = ctypes.c_int
    lib.minisgl_check_indices.argtypes = [vp, i32, i64, i32, vp, vp, i32, i32, vp, vp]
    lib.minisgl_check_indices.restype = ctypes.c_int
    lib.minisgl_last_error.argtypes = []
    lib.minisgl_last_error.restype = ctypes.c_char_p
    lib.minisgl_device_sm_count.argtypes = []
    lib.minisgl_device_sm_count.restype = i32
    lib.minisgl_debug_timeout_count.argtypes = [ctypes.POINTER(ctypes.c_uint32)]
    lib.minisgl_debug_timeout_count.restype = ctypes.c_int
    lib.minisgl_cascade_extend_workspace_bytes.argtypes = [i32, i32, i32]
    lib.minisgl_cascade_extend_workspace_bytes.restype = sz
    lib.minisgl_cascade_extend_attn.argtypes = [P, i32, vp, i32, vp, i32, i64, i32, vp, vp, vp, i32, i32,
                                                f32, vp, vp, sz, vp]
    lib.minisgl_cascade_extend_attn.restype = ctypes.c_int
    lib.minisgl_check_shared_prefix.argtypes = [vp, i32, i64, i32, i32, vp, vp, vp]
    lib.minisgl_check_shared_prefix.restype = ctypes.c_int
    lib.minisgl_debug_set_pdl.argtypes = [ctypes.c_int]
    lib.minisgl_debug_set_pdl.restype = ctypes.c_int
    _lib = lib
    return lib


def _check(rc: int, what: str) -> None:
    if rc != 0:
        msg = load_library().minisgl_last_error().decode(errors="replace")
        raise MinisglError(f"{what} failed ({rc}): {msg}")


def _stream(stream) -> ctypes.c_void_p:
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _rows_ok(t: torch.Tensor, n: int, row: int) -> bool:
    """True when t is [n, ...] and each t[i] is `row` contiguous elements
    (read from the shape and strides alone: indexing a tensor costs several
    microseconds of host time per call)."""
    if t.dim() < 2 or t.shape[0] != n:
        return False
    expect = 1
    for size, stride in zip(reversed(t.shape[1:]), reversed(t.stride()[1:])):
        if size != 1 and stride != expect:
            return False
        expect *= size
    return expect == row


def _need(t: torch.Tensor, name: str, dtype: torch.dtype) -> None:
    if not t.is_cuda:
        raise MinisglError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise MinisglError(f"{name} must be {dtype}, got {t.dtype}")


class KVPool:
    """A paged KV pool: one bf16 tensor of logical shape (2, L, R, H_kv, d).

    `tensor` may be LayerFirst (contiguous (2, L, R, H_kv, d)) or a permuted
    PageFirst view; only strides are read.  The pool is caller-owned device
    memory; the library keeps no reference to it."""

    def __init__(self, tensor: torch.Tensor, page_size: int = 1):
        if tensor.dim() != 5 or tensor.shape[0] != 2:
            raise MinisglError("pool tensor must have shape (2, L, R, H_kv, d)")
        _need(tensor, "pool", torch.bfloat16)
        if tensor.stride(4) != 1 or tensor.stride(3) != tensor.shape[4]:
            raise MinisglError("pool rows must be (H_kv, d) contiguous")
        self.tensor = tensor
        self.page_size = page_size
        _, L, R, H, d = tensor.shape
        self.num_layers, self.num_rows, self.num_kv_heads, self.head_dim = L, R, H, d
        self.desc = _PoolDesc(
            k_base=tensor[0].data_ptr(), v_base=tensor[1].data_ptr(),
            layer_stride=tensor.stride(1), row_stride=tensor.stride(2),
            num_layers=L, num_rows=R, num_kv_heads=H, head_dim=d, page_size=page_size,
            dtype=MINISGL_BF16)

    def k(self, layer: int) -> torch.Tensor:
        return self.tensor[0, layer]

    def v(self, layer: int) -> torch.Tensor:
        return self.tensor[1, layer]


def kv_pool_bytes(num_layers: int, num_kv_heads: int, head_dim: int, num_tokens: int,
                  elem_bytes: int = 2) -> int:
    """Bytes the pool needs to hold num_tokens token rows in every layer, K and V."""
    return 2 * num_layers * num_kv_heads * head_dim * num_tokens * elem_bytes


def minisgl_store_kv(pool: KVPool, layer: int, k: torch.Tensor, v: torch.Tensor,
                     out_loc: torch.Tensor, stream=None) -> None:
    """pool[K|V][layer][out_loc[i]] = k[i] | v[i] for every new token i (bit-exact)."""
    lib = load_library()
    _need(k, "k", torch.bfloat16)
    _need(v, "v", torch.bfloat16)
    _need(out_loc, "out_loc", torch.int32)
    n = out_loc.numel()
    row = pool.num_kv_heads * pool.head_dim
    for t, nm in ((k, "k"), (v, "v")):
        if not _rows_ok(t, n, row):
            raise MinisglError(f"{nm} must be [n_tokens, H_kv, d] with contiguous rows")
    if not out_loc.is_contiguous():
        raise MinisglError("out_loc must be contiguous")
    _check(lib.minisgl_store_kv(ctypes.byref(pool.desc), layer, _ptr(k), _ptr(v), k.stride(0),
                                v.stride(0), _ptr(out_loc), n, _stream(stream)), "store_kv")


def minisgl_decode_workspace_bytes(batch: int, num_q_heads: int, num_kv_heads: int, head_dim: int,
                                   max_splits: int = 16) -> int:
    return int(load_library().minisgl_decode_workspace_bytes(batch, num_q_heads, num_kv_heads,
                                                             head_dim, max_splits))


_ws_cache = {}


def decode_workspace(batch: int, num_q_heads: int, pool: KVPool, max_splits: int = 16,
                     device=None) -> torch.Tensor:
    """A workspace tensor for minisgl_decode_attn, cached per shape and device."""
    device = torch.device(device or pool.tensor.device)
    nbytes = minisgl_decode_workspace_bytes(batch, num_q_heads, pool.num_kv_heads, pool.head_dim,
                                            max_splits)
    key = (device, nbytes)
    ws = _ws_cache.get(key)
    if ws is None:
        ws = torch.empty(nbytes, dtype=torch.uint8, device=device)
        _ws_cache[key] = ws
    return ws


def minisgl_decode_attn(pool: KVPool, layer: int, q: torch.Tensor, page_table: torch.Tensor,
                        seq_lens: torch.Tensor, sm_scale: float, out: Optional[torch.Tensor] = None,
                        workspace: Optional[torch.Tensor] = None, split_tokens: int = 0,
                        max_splits: int = 16, stream=None) -> torch.Tensor:
    """Decode attention of q [B, H_q, d] over each request's page_table row."""
    lib = load_library()
    _need(q, "q", torch.bfloat16)
    _need(page_table, "page_table", torch.int32)
    _need(seq_lens, "seq_lens", torch.int32)
    B, Hq, d = q.shape
    if not q.is_contiguous() or d != pool.head_dim:
        raise MinisglError("q must be contiguous [B, H_q, head_dim]")
    if page_table.dim() != 2 or page_table.shape[0] != B or page_table.stride(1) != 1:
        raise MinisglError("page_table must be [B, W] with unit column stride")
    if seq_lens.numel() != B or not seq_lens.is_contiguous():
        raise MinisglError("seq_lens must be contiguous [B]")
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", torch.bfloat16)
    if workspace is None:
        workspace = decode_workspace(B, Hq, pool, max_splits)
    _check(lib.minisgl_decode_attn(ctypes.byref(pool.desc), layer, _ptr(q), Hq, _ptr(page_table), B,
                                   page_table.stride(0), page_table.shape[1], _ptr(seq_lens),
                                   float(sm_scale), _ptr(out), _ptr(workspace), workspace.numel(),
                                   split_tokens, _stream(stream)), "decode_attn")
    return out


def minisgl_decode_attn_noalloc(pool: KVPool, layer: int, q: torch.Tensor, page_table: torch.Tensor,
                                seq_lens: torch.Tensor, sm_scale: float,
                                out: Optional[torch.Tensor] = None, split_tokens: int = 0,
                                stream=None) -> torch.Tensor:
    """minisgl_decode_attn without a workspace, for callers that cannot allocate
    device memory: the split-KV scratch comes from a fixed 32 MiB array inside
    the library (one per GPU, shared by all calls, so calls must not overlap on
    the GPU).  `out` must be given by a caller that cannot allocate; when it is
    None this wrapper allocates it with torch for convenience."""
    lib = load_library()
    _need(q, "q", torch.bfloat16)
    _need(page_table, "page_table", torch.int32)
    _need(seq_lens, "seq_lens", torch.int32)
    B, Hq, d = q.shape
    if not q.is_contiguous() or d != pool.head_dim:
        raise MinisglError("q must be contiguous [B, H_q, head_dim]")
    if page_table.dim() != 2 or page_table.shape[0] != B or page_table.stride(1) != 1:
        raise MinisglError("page_table must be [B, W] with unit column stride")
    if seq_lens.numel() != B or not seq_lens.is_contiguous():
        raise MinisglError("seq_lens must be contiguous [B]")
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", torch.bfloat16)
    _check(lib.minisgl_decode_attn_noalloc(ctypes.byref(pool.desc), layer, _ptr(q), Hq,
                                           _ptr(page_table), B, page_table.stride(0),
                                           page_table.shape[1], _ptr(seq_lens), float(sm_scale),
                                           _ptr(out), split_tokens, _stream(stream)),
           "decode_attn_noalloc")
    return out


def minisgl_extend_attn(pool: KVPool, layer: int, q: torch.Tensor, page_table: torch.Tensor,
                        cached_lens: torch.Tensor, extend_lens: torch.Tensor,
                        q_offsets: torch.Tensor, sm_scale: float,
                        out: Optional[torch.Tensor] = None, work_counter: Optional[torch.Tensor] = None,
                        stream=None) -> torch.Tensor:
    """Causal extend attention of the packed new tokens q [T, H_q, d].
    work_counter: optional int32 CUDA tensor of 2 elements, zero before its
    first use (see extend_work_counter); calls that may run concurrently on
    different streams need different counters."""
    lib = load_library()
    _need(q, "q", torch.bfloat16)
    for t, nm in ((page_table, "page_table"), (cached_lens, "cached_lens"),
                  (extend_lens, "extend_lens"), (q_offsets, "q_offsets")):
        _need(t, nm, torch.int32)
    T, Hq, d = q.shape
    B = cached_lens.numel()
    if not q.is_contiguous() or d != pool.head_dim:
        raise MinisglError("q must be contiguous [T, H_q, head_dim]")
    if page_table.dim() != 2 or page_table.shape[0] != B or page_table.stride(1) != 1:
        raise MinisglError("page_table must be [B, W] with unit column stride")
    if extend_lens.numel() != B or q_offsets.numel() != B + 1:
        raise MinisglError("extend_lens must be [B] and q_offsets [B+1]")
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", torch.bfloat16)
    if work_counter is not None:
        _need(work_counter, "work_counter", torch.int32)
        if work_counter.numel() < 2 or not work_counter.is_contiguous():
            raise MinisglError("work_counter must be a contiguous int32 tensor of 2 elements")
    _check(lib.minisgl_extend_attn(ctypes.byref(pool.desc), layer, _ptr(q), Hq, _ptr(page_table), B,
                                   page_table.stride(0), page_table.shape[1], _ptr(cached_lens),
                                   _ptr(extend_lens), _ptr(q_offsets), T, float(sm_scale), _ptr(out),
                                   _ptr(work_counter), _stream(stream)), "extend_attn")
    return out


def extend_work_counter(device=None) -> torch.Tensor:
    """A zeroed work counter for minisgl_extend_attn (8 bytes of device memory)."""
    return torch.zeros(2, dtype=torch.int32, device=device or "cuda")


def minisgl_device_sm_count() -> int:
    return int(load_library().minisgl_device_sm_count())


def minisgl_check_indices(page_table: torch.Tensor, lens: torch.Tensor, num_rows: int,
                          out_loc: Optional[torch.Tensor] = None, counts: Optional[torch.Tensor] = None,
                          stream=None) -> torch.Tensor:
    """Count, on the device, the index values a decode or extend call over
    these tensors would read that lie outside the pool: returns an int32 CUDA
    tensor [page-table entries, out_loc entries, lengths outside
    [0, page_table width]] (read it after the stream).  lens is seq_lens for
    decode, cached_lens + extend_lens for extend."""
    lib = load_library()
    _need(page_table, "page_table", torch.int32)
    _need(lens, "lens", torch.int32)
    if page_table.dim() != 2 or page_table.stride(1) != 1:
        raise MinisglError("page_table must be [B, W] with unit column stride")
    if lens.numel() != page_table.shape[0] or not lens.is_contiguous():
        raise MinisglError("lens must be a contiguous [B] tensor")
    n_out = 0
    if out_loc is not None:
        _need(out_loc, "out_loc", torch.int32)
        if not out_loc.is_contiguous():
            raise MinisglError("out_loc must be contiguous")
        n_out = out_loc.numel()
    if counts is None:
        counts = torch.empty(3, dtype=torch.int32, device=page_table.device)
    _need(counts, "counts", torch.int32)
    if counts.numel() < 3:
        raise MinisglError("counts needs 3 elements")
    _check(lib.minisgl_check_indices(_ptr(page_table), page_table.shape[0], page_table.stride(0),
                                     page_table.shape[1], _ptr(lens), _ptr(out_loc), n_out,
                                     num_rows, _ptr(counts), _stream(stream)), "check_indices")
    return counts


def minisgl_debug_timeout_count() -> int:
    c = ctypes.c_uint32(0)
    _check(load_library().minisgl_debug_timeout_count(ctypes.byref(c)), "debug_timeout_count")
    return int(c.value)


def minisgl_debug_set_pdl(enabled: bool) -> bool:
    """Turn programmatic dependent launch on or off for the library's later
    launches (a measurement aid); returns the previous setting."""
    return bool(load_library().minisgl_debug_set_pdl(1 if enabled else 0))


def minisgl_rope_store_kv(pool: KVPool, layer: int, q: torch.Tensor, k: torch.Tensor,
                          v: torch.Tensor, positions: torch.Tensor, cos_sin_cache: torch.Tensor,
                          out_loc: torch.Tensor, stream=None) -> torch.Tensor:
    """Rotate q [N, H_q, d] in place and k [N, H_kv, d] into the pool by each
    token's position, and store v; returns q.  k is left unrotated."""
    lib = load_library()
    _need(q, "q", torch.bfloat16)
    _need(k, "k", torch.bfloat16)
    _need(v, "v", torch.bfloat16)
    _need(positions, "positions", torch.int32)
    _need(out_loc, "out_loc", torch.int32)
    _need(cos_sin_cache, "cos_sin_cache", torch.float32)
    n = out_loc.numel()
    d = pool.head_dim
    if q.dim() != 3 or q.shape[0] != n or q.shape[2] != d or q.stride(2) != 1 or q.stride(1) != d:
        raise MinisglError("q must be [n_tokens, H_q, head_dim] with contiguous rows")
    for t, nm in ((k, "k"), (v, "v")):
        if (t.dim() != 3 or t.shape[0] != n or t.shape[1] != pool.num_kv_heads or t.shape[2] != d
                or t.stride(2) != 1 or t.stride(1) != d):
            raise MinisglError(f"{nm} must be [n_tokens, H_kv, d] with contiguous rows")
    if positions.numel() != n or not positions.is_contiguous() or not out_loc.is_contiguous():
        raise MinisglError("positions and out_loc must be contiguous [n_tokens]")
    if cos_sin_cache.dim() != 2 or cos_sin_cache.shape[1] != d or not cos_sin_cache.is_contiguous():
        raise MinisglError("cos_sin_cache must be contiguous [max_positions, head_dim] float32")
    _check(lib.minisgl_rope_store_kv(ctypes.byref(pool.desc), layer, _ptr(q), q.shape[1], q.stride(0),
                                     _ptr(k), _ptr(v), k.stride(0), v.stride(0), _ptr(positions),
                                     _ptr(cos_sin_cache), cos_sin_cache.shape[0], _ptr(out_loc), n,
                                     _stream(stream)), "rope_store_kv")
    return q


def minisgl_cascade_workspace_bytes(batch: int, num_q_heads: int, num_kv_heads: int,
                                    head_dim: int) -> int:
    return int(load_library().minisgl_cascade_workspace_bytes(batch, num_q_heads, num_kv_heads,
                                                              head_dim))


def minisgl_cascade_decode_attn(pool: KVPool, layer: int, q: torch.Tensor, page_table: torch.Tensor,
                                seq_lens: torch.Tensor, shared_len: int, sm_scale: float,
                                out: Optional[torch.Tensor] = None,
                                workspace: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Decode attention of q [B, H_q, d] for requests whose first shared_len
    page-table entries are the same rows; the shared rows are read once."""
    lib = load_library()
    _need(q, "q", torch.bfloat16)
    _need(page_table, "page_table", torch.int32)
    _need(seq_lens, "seq_lens", torch.int32)
    B, Hq, d = q.shape
    if not q.is_contiguous() or d != pool.head_dim:
        raise MinisglError("q must be contiguous [B, H_q, head_dim]")
    if page_table.dim() != 2 or page_table.shape[0] != B or page_table.stride(1) != 1:
        raise MinisglError("page_table must be [B, W] with unit column stride")
    if seq_lens.numel() != B or not seq_lens.is_contiguous():
        raise MinisglError("seq_lens must be contiguous [B]")
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", torch.bfloat16)
    if workspace is None:
        nbytes = minisgl_cascade_workspace_bytes(B, Hq, pool.num_kv_heads, d)
        key = ("cascade", q.device, nbytes)
        workspace = _ws_cache.get(key)
        if workspace is None:
            # the first 256 bytes (a work counter) must start at zero
            workspace = torch.zeros(nbytes, dtype=torch.uint8, device=q.device)
            _ws_cache[key] = workspace
    _check(lib.minisgl_cascade_decode_attn(ctypes.byref(pool.desc), layer, _ptr(q), Hq, _ptr(page_table),
                                           B, page_table.stride(0), page_table.shape[1], _ptr(seq_lens),
                                           int(shared_len), float(sm_scale), _ptr(out), _ptr(workspace),
                                           workspace.numel(), _stream(stream)), "cascade_decode_attn")
    return out


def minisgl_store_decode_attn(pool: KVPool, layer: int, k: torch.Tensor, v: torch.Tensor,
                              out_loc: torch.Tensor, q: torch.Tensor, page_table: torch.Tensor,
                              seq_lens: torch.Tensor, sm_scale: float,
                              out: Optional[torch.Tensor] = None,
                              workspace: Optional[torch.Tensor] = None, split_tokens: int = 0,
                              max_splits: int = 16, stream=None) -> torch.Tensor:
    """minisgl_store_kv(k, v, out_loc) and minisgl_decode_attn in one pass
    (k, v: [B, H_kv, d], one new row per request)."""
    lib = load_library()
    for t, nm in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, nm, torch.bfloat16)
    for t, nm in ((page_table, "page_table"), (seq_lens, "seq_lens"), (out_loc, "out_loc")):
        _need(t, nm, torch.int32)
    B, Hq, d = q.shape
    if not q.is_contiguous() or d != pool.head_dim:
        raise MinisglError("q must be contiguous [B, H_q, head_dim]")
    row = pool.num_kv_heads * d
    for t, nm in ((k, "k"), (v, "v")):
        if not _rows_ok(t, B, row):
            raise MinisglError(f"{nm} must be [B, H_kv, d] with contiguous rows")
    if page_table.dim() != 2 or page_table.shape[0] != B or page_table.stride(1) != 1:
        raise MinisglError("page_table must be [B, W] with unit column stride")
    if seq_lens.numel() != B or not seq_lens.is_contiguous() or out_loc.numel() != B \
            or not out_loc.is_contiguous():
        raise MinisglError("seq_lens and out_loc must be contiguous [B]")
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", torch.bfloat16)
    if workspace is None:
        workspace = decode_workspace(B, Hq, pool, max_splits)
    _check(lib.minisgl_store_decode_attn(ctypes.byref(pool.desc), layer, _ptr(k), _ptr(v), k.stride(0),
                                         v.stride(0), _ptr(out_loc), _ptr(q), Hq, _ptr(page_table), B,
                                         page_table.stride(0), page_table.shape[1], _ptr(seq_lens),
                                         float(sm_scale), _ptr(out), _ptr(workspace), workspace.numel(),
                                         split_tokens, _stream(stream)), "store_decode_attn")
    return out


def minisgl_cascade_extend_workspace_bytes(total_q_tokens: int, num_q_heads: int, head_dim: int) -> int:
    return int(load_library().minisgl_cascade_extend_workspace_bytes(total_q_tokens, num_q_heads,
                                                                     head_dim))


def minisgl_cascade_extend_attn(pool: KVPool, layer: int, q: torch.Tensor, page_table: torch.Tensor,
                                cached_lens: torch.Tensor, extend_lens: torch.Tensor,
                                q_offsets: torch.Tensor, shared_len: int, sm_scale: float,
                                out: Optional[torch.Tensor] = None,
                                workspace: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Causal extend attention of q [T, H_q, d] for requests whose first
    shared_len page-table entries are the same rows: a pass of all new tokens
    against the shared rows, then each request's own rows with that pass's
    partial folded in."""
    lib = load_library()
    _need(q, "q", torch.bfloat16)
    for t, nm in ((page_table, "page_table"), (cached_lens, "cached_lens"),
                  (extend_lens, "extend_lens"), (q_offsets, "q_offsets")):
        _need(t, nm, torch.int32)
    T, Hq, d = q.shape
    B = cached_lens.numel()
    if not q.is_contiguous() or d != pool.head_dim:
        raise MinisglError("q must be contiguous [T, H_q, head_dim]")
    if page_table.dim() != 2 or page_table.shape[0] != B or page_table.stride(1) != 1:
        raise MinisglError("page_table must be [B, W] with unit column stride")
    if extend_lens.numel() != B or q_offsets.numel() != B + 1:
        raise MinisglError("extend_lens must be [B] and q_offsets [B+1]")
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", torch.bfloat16)
    if workspace is None:
        nbytes = minisgl_cascade_extend_workspace_bytes(T, Hq, d)
        key = ("cascade_extend", q.device, nbytes)
        workspace = _ws_cache.get(key)
        if workspace is None:
            # the first 256 bytes (a work counter) must start at zero
            workspace = torch.zeros(nbytes, dtype=torch.uint8, device=q.device)
            _ws_cache[key] = workspace
    _check(lib.minisgl_cascade_extend_attn(ctypes.byref(pool.desc), layer, _ptr(q), Hq, _ptr(page_table), B,
                                           page_table.stride(0), page_table.shape[1], _ptr(cached_lens),
                                           _ptr(extend_lens), _ptr(q_offsets), T, int(shared_len),
                                           float(sm_scale), _ptr(out), _ptr(workspace), workspace.numel(),
                                           _stream(stream)), "cascade_extend_attn")
    return out


def minisgl_check_shared_prefix(page_table: torch.Tensor, lens: torch.Tensor, shared_len: int,
                                counts: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Count, on the device, the shared-prefix page-table entries that differ
    from the first request's and the requests shorter than shared_len:
    returns an int32 CUDA tensor [differing entries, short requests] (read it
    after the stream).  lens: seq_lens for decode, cached_lens for extend."""
    lib = load_library()
    _need(page_table, "page_table", torch.int32)
    _need(lens, "lens", torch.int32)
    if page_table.dim() != 2 or page_table.stride(1) != 1:
        raise MinisglError("page_table must be [B, W] with unit column stride")
    if lens.numel() != page_table.shape[0] or not lens.is_contiguous():
        raise MinisglError("lens must be a contiguous [B] tensor")
    if counts is None:
        counts = torch.empty(2, dtype=torch.int32, device=page_table.device)
    _need(counts, "counts", torch.int32)
    if counts.numel() < 2:
        raise MinisglError("counts needs 2 elements")
    _check(lib.minisgl_check_shared_prefix(_ptr(page_table), page_table.shape[0], page_table.stride(0),
                                           page_table.shape[1], int(shared_len), _ptr(lens), _ptr(counts),
                                           _stream(stream)), "check_shared_prefix")
    return counts
