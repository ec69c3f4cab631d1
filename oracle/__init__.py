"""fp64 CPU oracle for attention over a paged KV pool -- TEST INFRASTRUCTURE.

Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline leg may import
this package.  The product library never does; the two share no code.

The arithmetic lives in oracle.c (plain C, double precision, one thread); this
module compiles it with gcc and marshals numpy arrays through ctypes.  bf16
tensors are passed as their raw 16-bit patterns and widened exactly to double
inside the C code.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "oracle.c")
LIB_DIR = os.path.join(_HERE, "_lib")
LIB_PATH = os.path.join(LIB_DIR, "liboracle.so")


def compile_oracle(source: str = SOURCE, out: str = LIB_PATH) -> str:
    """Compile an oracle C source into a shared library (plain gcc, no fast-math)."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    if (os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(source)
            and source == SOURCE):
        return out
    tmp = out + ".tmp%d" % os.getpid()
    subprocess.run(["gcc", "-std=c11", "-O2", "-fPIC", "-shared", "-o", tmp, source, "-lm"],
                   check=True)
    os.replace(tmp, out)
    return out


def _u16(a) -> np.ndarray:
    """bf16 torch tensor or uint16 numpy array -> contiguous uint16 numpy array."""
    try:
        import torch
        if isinstance(a, torch.Tensor):
            assert a.dtype == torch.bfloat16, a.dtype
            return a.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
    except ImportError:  # pragma: no cover
        pass
    a = np.ascontiguousarray(a)
    assert a.dtype == np.uint16, a.dtype
    return a


def _i32(a) -> np.ndarray:
    try:
        import torch
        if isinstance(a, torch.Tensor):
            a = a.detach().cpu().numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(a, dtype=np.int32)


def _p(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


class Oracle:
    """ctypes front end of one compiled oracle library."""

    def __init__(self, lib_path: Optional[str] = None):
        self.path = lib_path or compile_oracle()
        self.lib = ctypes.CDLL(self.path)
        vp, i32, i64, dbl = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_double
        self.lib.oracle_store_kv.argtypes = [vp, vp, i64, i64, vp, vp, i64, vp, i64, i64]
        self.lib.oracle_store_kv.restype = ctypes.c_int
        self.lib.oracle_decode.argtypes = [vp, i32, i32, i32, i32, vp, vp, i64, i64, vp, i64, vp,
                                           vp, dbl, vp, vp]
        self.lib.oracle_decode.restype = ctypes.c_int
        self.lib.oracle_extend.argtypes = [vp, i32, i32, i32, i32, vp, vp, i64, i64, vp, i64, vp,
                                           vp, dbl, vp]
        self.lib.oracle_extend.restype = ctypes.c_int
        self.lib.oracle_lse_merge.argtypes = [i64, i64, i32, vp, vp, vp, vp]
        self.lib.oracle_lse_merge.restype = None
        self.lib.oracle_rope.argtypes = [vp, i64, i32, i32, vp, vp, i64, vp]
        self.lib.oracle_rope.restype = ctypes.c_int

    # -- store_kv ---------------------------------------------------------
    def store_kv(self, k_pool: np.ndarray, v_pool: np.ndarray, k, v, out_loc) -> None:
        """In place on uint16 pools shaped [R, H_kv, d] (or [R, row_elems]).
        k, v: [N, H_kv, d] bf16 / uint16; out_loc: [N] int32."""
        assert k_pool.dtype == np.uint16 and k_pool.flags.c_contiguous
        assert v_pool.dtype == np.uint16 and v_pool.flags.c_contiguous
        k, v, loc = _u16(k), _u16(v), _i32(out_loc)
        R = k_pool.shape[0]
        row = int(np.prod(k_pool.shape[1:]))
        n = loc.shape[0]
        rc = self.lib.oracle_store_kv(_p(k_pool), _p(v_pool), row, R, _p(k), _p(v), row, _p(loc),
                                      n, row)
        if rc != 0:
            raise ValueError("oracle_store_kv: out_loc outside the pool")

    # -- decode -----------------------------------------------------------
    def decode(self, q, k_pool, v_pool, page_table, seq_lens, sm_scale: float, j_begin=None):
        """q [B, H_q, d]; pools [R, H_kv, d]; page_table [B, W]; seq_lens [B].
        Returns (out [B, H_q, d] float64, lse [B, H_q] float64).  With j_begin,
        request r covers logical tokens [j_begin[r], seq_lens[r]) only."""
        q, kp, vp = _u16(q), _u16(k_pool), _u16(v_pool)
        pt, sl = _i32(page_table), _i32(seq_lens)
        jb = None if j_begin is None else _i32(j_begin)
        B, Hq, d = q.shape
        R, Hk = kp.shape[0], kp.shape[1]
        out = np.zeros((B, Hq, d), dtype=np.float64)
        lse = np.zeros((B, Hq), dtype=np.float64)
        rc = self.lib.oracle_decode(_p(q), B, Hq, Hk, d, _p(kp), _p(vp), Hk * d, R, _p(pt),
                                    pt.shape[1], _p(jb), _p(sl), float(sm_scale), _p(out), _p(lse))
        if rc != 0:
            raise ValueError("oracle_decode: bad arguments or row index")
        return out, lse

    # -- extend -----------------------------------------------------------
    def extend(self, q, k_pool, v_pool, page_table, cached_lens, extend_lens, sm_scale: float):
        """q [T, H_q, d] packed in request order; returns out [T, H_q, d] float64."""
        q, kp, vp = _u16(q), _u16(k_pool), _u16(v_pool)
        pt, cl, el = _i32(page_table), _i32(cached_lens), _i32(extend_lens)
        T, Hq, d = q.shape
        R, Hk = kp.shape[0], kp.shape[1]
        assert int(el.sum()) == T
        out = np.zeros((T, Hq, d), dtype=np.float64)
        rc = self.lib.oracle_extend(_p(q), cl.shape[0], Hq, Hk, d, _p(kp), _p(vp), Hk * d, R,
                                    _p(pt), pt.shape[1], _p(cl), _p(el), float(sm_scale), _p(out))
        if rc != 0:
            raise ValueError("oracle_extend: bad arguments or row index")
        return out

    # -- lse merge --------------------------------------------------------
    def lse_merge(self, o_parts: np.ndarray, lse_parts: np.ndarray):
        """o_parts [S, ..., d], lse_parts [S, ...] -> (o [..., d], lse [...])."""
        o_parts = np.ascontiguousarray(o_parts, dtype=np.float64)
        lse_parts = np.ascontiguousarray(lse_parts, dtype=np.float64)
        S, d = o_parts.shape[0], o_parts.shape[-1]
        vec_shape = lse_parts.shape[1:]
        n_vec = int(np.prod(vec_shape)) if vec_shape else 1
        out = np.zeros(vec_shape + (d,), dtype=np.float64)
        lse = np.zeros(vec_shape, dtype=np.float64)
        self.lib.oracle_lse_merge(S, n_vec, d, _p(o_parts), _p(lse_parts), _p(out), _p(lse))
        return out, lse

    # -- rope -------------------------------------------------------------
    def rope(self, x, positions, cos_sin_cache):
        """x [N, H, d] bf16 / uint16; positions [N] int32; cos_sin_cache
        [max_positions, d] float32 ([cos | sin] per row).  Returns the rotated
        x as float64 [N, H, d]."""
        xs = _u16(x)
        pos = _i32(positions)
        try:
            import torch
            if isinstance(cos_sin_cache, torch.Tensor):
                cos_sin_cache = cos_sin_cache.detach().cpu().numpy()
        except ImportError:  # pragma: no cover
            pass
        cache = np.ascontiguousarray(cos_sin_cache, dtype=np.float32)
        N, H, d = xs.shape
        assert cache.shape[1] == d and pos.shape[0] == N
        out = np.zeros((N, H, d), dtype=np.float64)
        rc = self.lib.oracle_rope(_p(xs), N, H, d, _p(pos), _p(cache), cache.shape[0], _p(out))
        if rc != 0:
            raise ValueError("oracle_rope: position outside the cache or odd head_dim")
        return out


_default: Optional[Oracle] = None


def get() -> Oracle:
    global _default
    if _default is None:
        _default = Oracle()
    return _default
