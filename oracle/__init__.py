"""fp64 CPU oracle for paged MLA decode (test infrastructure).

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package; the library itself never does.  The arithmetic
lives in ``mla_oracle.c`` (plain C, fp64); this module compiles it with gcc and
marshals numpy arrays into it.

Definition followed: scaled-dot-product attention of every query row over
the latent cache rows it may see (bottom-right causal inside the ``s_q`` query
tokens), values = the first 512 dims of the same row, lse = natural log of
the softmax denominator of the scaled logits.  Sparse decode (one query
token per entry) is the same attention over the cache rows at a listed set of
token positions.  The header of ``mla_oracle.c`` states both in full.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import sys

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "mla_oracle.c")
_LIB = os.path.join(_HERE, "_build", "libmla_oracle.so")

D_V = 512


def compile_source(src: str, lib_path: str) -> str:
    """Compile one oracle source file with gcc into ``lib_path``."""
    os.makedirs(os.path.dirname(lib_path), exist_ok=True)
    tmp = lib_path + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                           "-o", tmp, src, "-lm"])
    os.replace(tmp, lib_path)
    return lib_path


def build(force: bool = False) -> str:
    """Compile the oracle (plain C, no target-specific flags)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(SOURCE):
        compile_source(SOURCE, _LIB)
    return _LIB


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def _c(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a, a.ctypes.data_as(ctypes.c_void_p)


class Oracle:
    """ctypes front end of one compiled oracle library."""

    def __init__(self, lib_path: str):
        lib = ctypes.CDLL(lib_path)
        P, I = ctypes.c_void_p, ctypes.c_int
        lib.oracle_mla_decode_rows.argtypes = [P, P, I, P, I, P, I, I, I, ctypes.c_double, I, P,
                                               I, I, P, P, I]
        lib.oracle_mla_decode_rows.restype = I
        lib.oracle_mla_decode.argtypes = [P, P, I, P, I, P, I, I, I, ctypes.c_double, P, P, I]
        lib.oracle_mla_decode.restype = I
        lib.oracle_mla_decode_sparse_rows.argtypes = [P, P, I, P, I, P, P, I, P, I, I,
                                                      ctypes.c_double, I, P, I, I, P, P, I]
        lib.oracle_mla_decode_sparse_rows.restype = I
        lib.oracle_lse_combine.argtypes = [I, P, P, P, P]
        lib.oracle_lse_combine.restype = None
        self.lib = lib

    def mla_decode(self, inp, nthreads: int | None = None, scale: float | None = None):
        """All rows: returns (out [B,s_q,h_q,512] f64, lse [B,h_q,s_q] f64)."""
        B, s_q, h_q = inp.batch, inp.s_q, inp.h_q
        _q, qp = _c(inp.q, np.uint16)
        _kv, kvp = _c(inp.kv_cache, np.uint16)
        _bt, btp = _c(inp.block_table, np.int32)
        _sl, slp = _c(inp.cache_seqlens, np.int32)
        out = np.zeros((B, s_q, h_q, D_V), dtype=np.float64)
        lse = np.zeros((B, h_q, s_q), dtype=np.float64)
        rc = self.lib.oracle_mla_decode(
            qp, kvp, inp.num_pages, btp, inp.max_pages, slp, B, s_q, h_q,
            float(inp.softmax_scale if scale is None else scale),
            out.ctypes.data_as(ctypes.c_void_p), lse.ctypes.data_as(ctypes.c_void_p),
            nthreads or default_threads())
        if rc != 0:
            raise ValueError("oracle: index out of range")
        return out, lse

    def mla_decode_rows(self, inp, rows, key_begin: int = 0, key_end: int = 2**31 - 1,
                        nthreads: int | None = None, scale: float | None = None):
        """Selected rows (array of (b, i, h)); returns (out [n,512], lse [n])."""
        rows_a, rp = _c(np.asarray(rows, dtype=np.int32).reshape(-1, 3), np.int32)
        n = rows_a.shape[0]
        _q, qp = _c(inp.q, np.uint16)
        _kv, kvp = _c(inp.kv_cache, np.uint16)
        _bt, btp = _c(inp.block_table, np.int32)
        _sl, slp = _c(inp.cache_seqlens, np.int32)
        out = np.zeros((n, D_V), dtype=np.float64)
        lse = np.zeros((n,), dtype=np.float64)
        rc = self.lib.oracle_mla_decode_rows(
            qp, kvp, inp.num_pages, btp, inp.max_pages, slp, inp.batch, inp.s_q, inp.h_q,
            float(inp.softmax_scale if scale is None else scale), n, rp, int(key_begin),
            int(key_end), out.ctypes.data_as(ctypes.c_void_p),
            lse.ctypes.data_as(ctypes.c_void_p), nthreads or default_threads())
        if rc != 0:
            raise ValueError("oracle: index out of range")
        return out, lse

    def mla_decode_sparse_rows(self, si, rows_bh, key_begin: int = 0, key_end: int = 2**31 - 1,
                               nthreads: int | None = None, scale: float | None = None):
        """Sparse decode of selected (b, h) rows: returns (out [n,512], lse [n]).
        key_begin/key_end restrict the positions in each entry's index list."""
        inp = si.base
        rows_a, rp = _c(np.asarray(rows_bh, dtype=np.int32).reshape(-1, 2), np.int32)
        n = rows_a.shape[0]
        _q, qp = _c(inp.q, np.uint16)
        _kv, kvp = _c(inp.kv_cache, np.uint16)
        _bt, btp = _c(inp.block_table, np.int32)
        _sl, slp = _c(inp.cache_seqlens, np.int32)
        _ix, ixp = _c(si.indices, np.int32)
        _ct, ctp = _c(si.counts, np.int32)
        out = np.zeros((n, D_V), dtype=np.float64)
        lse = np.zeros((n,), dtype=np.float64)
        rc = self.lib.oracle_mla_decode_sparse_rows(
            qp, kvp, inp.num_pages, btp, inp.max_pages, slp, ixp, si.indices.shape[1], ctp,
            inp.batch, inp.h_q, float(inp.softmax_scale if scale is None else scale), n, rp,
            int(key_begin), int(key_end), out.ctypes.data_as(ctypes.c_void_p),
            lse.ctypes.data_as(ctypes.c_void_p), nthreads or default_threads())
        if rc != 0:
            raise ValueError("oracle: index or count out of range")
        return out, lse

    def mla_decode_sparse(self, si, nthreads: int | None = None, scale: float | None = None):
        """Sparse decode, every row: returns (out [B,1,h_q,512], lse [B,h_q,1])."""
        B, h_q = si.base.batch, si.base.h_q
        rows = np.array([(b, h) for b in range(B) for h in range(h_q)], dtype=np.int32)
        out, lse = self.mla_decode_sparse_rows(si, rows, nthreads=nthreads, scale=scale)
        return out.reshape(B, 1, h_q, D_V), lse.reshape(B, h_q, 1)

    def lse_combine(self, lse_parts, o_parts):
        """Merge results over disjoint key sets: returns (lse, out[512])."""
        _l, lp = _c(np.asarray(lse_parts, dtype=np.float64).reshape(-1), np.float64)
        _o, op = _c(np.asarray(o_parts, dtype=np.float64).reshape(-1, D_V), np.float64)
        out = np.zeros(D_V, dtype=np.float64)
        lse = np.zeros(1, dtype=np.float64)
        self.lib.oracle_lse_combine(_l.shape[0], lp, op, lse.ctypes.data_as(ctypes.c_void_p),
                                    out.ctypes.data_as(ctypes.c_void_p))
        return float(lse[0]), out


_default: Oracle | None = None


def default() -> Oracle:
    global _default
    if _default is None:
        _default = Oracle(build())
    return _default


def mla_decode(inp, nthreads=None, scale=None):
    return default().mla_decode(inp, nthreads, scale)


def mla_decode_rows(inp, rows, key_begin=0, key_end=2**31 - 1, nthreads=None, scale=None):
    return default().mla_decode_rows(inp, rows, key_begin, key_end, nthreads, scale)


def lse_combine(lse_parts, o_parts):
    return default().lse_combine(lse_parts, o_parts)


def mla_decode_sparse(si, nthreads=None, scale=None):
    return default().mla_decode_sparse(si, nthreads, scale)


def mla_decode_sparse_rows(si, rows_bh, key_begin=0, key_end=2**31 - 1, nthreads=None,
                           scale=None):
    return default().mla_decode_sparse_rows(si, rows_bh, key_begin, key_end, nthreads, scale)


if __name__ == "__main__":  # pragma: no cover
    print(build(force="--force" in sys.argv))
