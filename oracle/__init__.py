"""fp64 CPU oracles for paged MLA decode and its neighbouring steps (test infrastructure).

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

``attention_oracle.c`` is dense scaled-dot-product attention (causal or
not) over [B, S, H, d] tensors, the result a FlashAttention kernel computes.
``prologue_oracle.c`` writes out the two steps that prepare a decode call
(the new tokens' rows appended to the paged cache, bit for bit; the query
absorbed through W_UK, in fp64) and ``gemm_oracle.c`` the plain matrix
product C = A B of the tensor-core GEMM, in fp64 from fp16 or bf16 inputs.
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
PROLOGUE_SOURCE = os.path.join(_HERE, "prologue_oracle.c")
_PROLOGUE_LIB = os.path.join(_HERE, "_build", "libprologue_oracle.so")
GEMM_SOURCE = os.path.join(_HERE, "gemm_oracle.c")
_GEMM_LIB = os.path.join(_HERE, "_build", "libgemm_oracle.so")
ATTENTION_SOURCE = os.path.join(_HERE, "attention_oracle.c")
_ATTENTION_LIB = os.path.join(_HERE, "_build", "libattention_oracle.so")

D_V = 512


def compile_source(src: str, lib_path: str) -> str:
    """Compile one oracle source file with gcc into ``lib_path``."""
    os.makedirs(os.path.dirname(lib_path), exist_ok=True)
    tmp = lib_path + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                           "-o", tmp, src, "-lm"])
    os.replace(tmp, lib_path)
    return lib_path


def _build_one(src: str, lib: str, force: bool) -> str:
    if force or not os.path.exists(lib) or os.path.getmtime(lib) < os.path.getmtime(src):
        compile_source(src, lib)
    return lib


def build(force: bool = False) -> str:
    """Compile the oracles (plain C, no target-specific flags); returns the
    decode oracle's library."""
    _build_one(PROLOGUE_SOURCE, _PROLOGUE_LIB, force)
    _build_one(GEMM_SOURCE, _GEMM_LIB, force)
    _build_one(ATTENTION_SOURCE, _ATTENTION_LIB, force)
    return _build_one(SOURCE, _LIB, force)


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


class Prologue:
    """ctypes front end of the cache-append / query-absorption oracle."""

    def __init__(self, lib_path: str):
        lib = ctypes.CDLL(lib_path)
        P, I = ctypes.c_void_p, ctypes.c_int
        lib.oracle_cache_append.argtypes = [P, P, I, P, I, P, I, I]
        lib.oracle_cache_append.restype = I
        lib.oracle_q_absorb.argtypes = [P, P, I, I, I, I, P]
        lib.oracle_q_absorb.restype = None
        self.lib = lib

    def cache_append(self, kv_new, kv_cache, block_table, cache_seqlens):
        """Returns a copy of kv_cache (uint16 [pages, 64, 1, 576]) with the new
        rows (uint16 [B, s_q, 576]) written at positions L_b - s_q + i."""
        kv_new = np.ascontiguousarray(kv_new, dtype=np.uint16)
        B, s_q = int(kv_new.shape[0]), int(kv_new.shape[1])
        cache = np.array(kv_cache, dtype=np.uint16, copy=True, order="C")
        _n, np_ = _c(kv_new, np.uint16)
        _bt, btp = _c(block_table, np.int32)
        _sl, slp = _c(cache_seqlens, np.int32)
        rc = self.lib.oracle_cache_append(np_, cache.ctypes.data_as(ctypes.c_void_p),
                                          int(cache.shape[0]), btp, int(_bt.shape[1]), slp, B,
                                          s_q)
        if rc != 0:
            raise ValueError("oracle: new token position or page out of range")
        return cache

    def q_absorb(self, q_nope, w_uk):
        """q_nope uint16 [B, s_q, h_q, d_nope], w_uk uint16 [h_q, d_nope, d_c]
        -> fp64 [B, s_q, h_q, d_c]."""
        q_nope = np.ascontiguousarray(q_nope, dtype=np.uint16)
        B, s_q, h_q, dn = (int(x) for x in q_nope.shape)
        w_uk = np.ascontiguousarray(w_uk, dtype=np.uint16)
        assert w_uk.shape[0] == h_q and w_uk.shape[1] == dn
        dc = int(w_uk.shape[2])
        out = np.zeros((B, s_q, h_q, dc), dtype=np.float64)
        self.lib.oracle_q_absorb(q_nope.ctypes.data_as(ctypes.c_void_p),
                                 w_uk.ctypes.data_as(ctypes.c_void_p), B * s_q, h_q, dn, dc,
                                 out.ctypes.data_as(ctypes.c_void_p))
        return out


class Gemm:
    """ctypes front end of the GEMM oracle (fmt 0: fp16 inputs, 1: bf16)."""

    def __init__(self, lib_path: str):
        lib = ctypes.CDLL(lib_path)
        P, I = ctypes.c_void_p, ctypes.c_int
        lib.oracle_gemm.argtypes = [P, P, I, I, I, I, P, I]
        lib.oracle_gemm.restype = I
        lib.oracle_gemm_entries.argtypes = [P, P, I, I, I, I, I, P, P, I]
        lib.oracle_gemm_entries.restype = I
        self.lib = lib

    def gemm(self, a_bits, b_bits, fmt: int, nthreads: int | None = None):
        """a_bits uint16 [M, K], b_bits uint16 [K, N] -> C fp64 [M, N]."""
        a = np.ascontiguousarray(a_bits, dtype=np.uint16)
        b = np.ascontiguousarray(b_bits, dtype=np.uint16)
        M, K = a.shape
        K2, N = b.shape
        assert K == K2
        c = np.zeros((M, N), dtype=np.float64)
        self.lib.oracle_gemm(a.ctypes.data_as(ctypes.c_void_p), b.ctypes.data_as(ctypes.c_void_p),
                             M, N, K, int(fmt), c.ctypes.data_as(ctypes.c_void_p),
                             nthreads or default_threads())
        return c

    def gemm_entries(self, a_bits, b_bits, fmt: int, entries, nthreads: int | None = None):
        """Selected entries (array of (m, n)) of C = A B, fp64 [n]."""
        a = np.ascontiguousarray(a_bits, dtype=np.uint16)
        b = np.ascontiguousarray(b_bits, dtype=np.uint16)
        M, K = a.shape
        N = b.shape[1]
        e = np.ascontiguousarray(np.asarray(entries, dtype=np.int32).reshape(-1, 2))
        out = np.zeros(e.shape[0], dtype=np.float64)
        rc = self.lib.oracle_gemm_entries(a.ctypes.data_as(ctypes.c_void_p),
                                          b.ctypes.data_as(ctypes.c_void_p), M, N, K, int(fmt),
                                          int(e.shape[0]), e.ctypes.data_as(ctypes.c_void_p),
                                          out.ctypes.data_as(ctypes.c_void_p),
                                          nthreads or default_threads())
        if rc != 0:
            raise ValueError("oracle: GEMM entry out of range")
        return out


class Attention:
    """ctypes front end of the dense attention oracle."""

    def __init__(self, lib_path: str):
        lib = ctypes.CDLL(lib_path)
        P, I, D = ctypes.c_void_p, ctypes.c_int, ctypes.c_double
        lib.oracle_attention.argtypes = [P, P, P, I, I, I, I, I, I, D, P, P, I]
        lib.oracle_attention.restype = I
        lib.oracle_attention_rows.argtypes = [P, P, P, I, I, I, I, I, I, D, I, P, P, P, I]
        lib.oracle_attention_rows.restype = I
        self.lib = lib

    @staticmethod
    def _shapes(ai):
        B, S, H, dqk = (int(x) for x in ai.q.shape)
        return B, S, H, dqk, int(ai.v.shape[3])

    def attention(self, ai, nthreads: int | None = None):
        """Every row: out fp64 [B, S, H, d_v], lse fp64 [B, H, S]."""
        B, S, H, dqk, dv = self._shapes(ai)
        _q, qp = _c(ai.q, np.uint16)
        _k, kp = _c(ai.k, np.uint16)
        _v, vp = _c(ai.v, np.uint16)
        out = np.zeros((B, S, H, dv), dtype=np.float64)
        lse = np.zeros((B, H, S), dtype=np.float64)
        self.lib.oracle_attention(qp, kp, vp, B, S, H, dqk, dv, int(ai.causal), float(ai.scale),
                                  out.ctypes.data_as(ctypes.c_void_p),
                                  lse.ctypes.data_as(ctypes.c_void_p),
                                  nthreads or default_threads())
        return out, lse

    def attention_rows(self, ai, rows, nthreads: int | None = None):
        """Selected rows (array of (b, h, i)): out [n, d_v], lse [n]."""
        B, S, H, dqk, dv = self._shapes(ai)
        r = np.ascontiguousarray(np.asarray(rows, dtype=np.int32).reshape(-1, 3))
        _q, qp = _c(ai.q, np.uint16)
        _k, kp = _c(ai.k, np.uint16)
        _v, vp = _c(ai.v, np.uint16)
        out = np.zeros((r.shape[0], dv), dtype=np.float64)
        lse = np.zeros((r.shape[0],), dtype=np.float64)
        rc = self.lib.oracle_attention_rows(qp, kp, vp, B, S, H, dqk, dv, int(ai.causal),
                                            float(ai.scale), int(r.shape[0]),
                                            r.ctypes.data_as(ctypes.c_void_p),
                                            out.ctypes.data_as(ctypes.c_void_p),
                                            lse.ctypes.data_as(ctypes.c_void_p),
                                            nthreads or default_threads())
        if rc != 0:
            raise ValueError("oracle: attention row out of range")
        return out, lse


_default: Oracle | None = None
_attention: Attention | None = None
_prologue: Prologue | None = None
_gemm: Gemm | None = None


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


def prologue() -> Prologue:
    global _prologue
    if _prologue is None:
        build()
        _prologue = Prologue(_PROLOGUE_LIB)
    return _prologue


def gemm_oracle() -> Gemm:
    global _gemm
    if _gemm is None:
        build()
        _gemm = Gemm(_GEMM_LIB)
    return _gemm


def attention_oracle() -> Attention:
    global _attention
    if _attention is None:
        build()
        _attention = Attention(_ATTENTION_LIB)
    return _attention


def attention(ai, nthreads=None):
    return attention_oracle().attention(ai, nthreads)


def attention_rows(ai, rows, nthreads=None):
    return attention_oracle().attention_rows(ai, rows, nthreads)


def cache_append(kv_new, kv_cache, block_table, cache_seqlens):
    return prologue().cache_append(kv_new, kv_cache, block_table, cache_seqlens)


def q_absorb(q_nope, w_uk):
    return prologue().q_absorb(q_nope, w_uk)


def gemm(a_bits, b_bits, fmt, nthreads=None):
    return gemm_oracle().gemm(a_bits, b_bits, fmt, nthreads)


def gemm_entries(a_bits, b_bits, fmt, entries, nthreads=None):
    return gemm_oracle().gemm_entries(a_bits, b_bits, fmt, entries, nthreads)


if __name__ == "__main__":  # pragma: no cover
    print(build(force="--force" in sys.argv))
