"""ctypes binding of libmla (the C ABI in include/mla.h).

Argument marshalling only: every step of the decode runs in the library's
CUDA kernels.  Device buffers are torch tensors (their data pointers are
passed through); torch is used for memory and streams, nothing else.  The
library must have been built (``__graft_entry__.build()`` or
``python -m mla_decode_attention_07_gb300.build``); loading fails loudly
otherwise, and on a device that is not sm_103 the calls return
MLA_ERR_UNSUPPORTED_DEVICE.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libmla.so")

MLA_OK = 0
MLA_ERR_INVALID_ARG = -1
MLA_ERR_WORKSPACE = -2
MLA_ERR_CUDA = -3
MLA_ERR_DEVICE_TIMEOUT = -4
MLA_ERR_DEVICE_BOUNDS = -5
MLA_ERR_UNSUPPORTED_DEVICE = -6
MLA_ERR_PLAN = -7

EXPORTED = ["mla_num_clusters", "mla_plan_size", "mla_plan_size_for_clusters",
            "mla_workspace_size", "mla_decode_plan", "mla_decode_plan_host", "mla_decode",
            "mla_decode_f32", "mla_decode_attend", "mla_decode_combine", "mla_decode_noalloc",
            "mla_decode_sparse", "mla_decode_sparse_f32", "mla_selftest_wait_timeout",
            "mla_check_device_error", "mla_strerror", "mla_cache_append", "mla_q_absorb",
            "mla_gemm", "mla_attention_fwd", "mla_decode_kernel_kind"]

MLA_DTYPE_F16 = 0
MLA_DTYPE_BF16 = 1
MLA_DTYPE_F32 = 2

_lib = None


class MlaError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {mla_strerror(code)} ({code})")


def load(path: str | None = None) -> ctypes.CDLL:
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"libmla is not built ({p} missing): run __graft_entry__.build()")
    lib = ctypes.CDLL(p)
    V, I, Z, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_float
    lib.mla_num_clusters.argtypes = [I]
    lib.mla_num_clusters.restype = I
    lib.mla_decode_kernel_kind.argtypes = [I, I, I, I, I]
    lib.mla_decode_kernel_kind.restype = I
    lib.mla_plan_size.argtypes = [I, I, I, I]
    lib.mla_plan_size.restype = Z
    lib.mla_plan_size_for_clusters.argtypes = [I, I, I, I]
    lib.mla_plan_size_for_clusters.restype = Z
    lib.mla_workspace_size.argtypes = [I, I, I, I]
    lib.mla_workspace_size.restype = Z
    lib.mla_decode_plan.argtypes = [V, I, I, I, V, Z, V]
    lib.mla_decode_plan.restype = I
    lib.mla_decode_plan_host.argtypes = [V, I, I, I, I, V, Z]
    lib.mla_decode_plan_host.restype = I
    lib.mla_decode.argtypes = [V, V, I, V, I, V, I, I, I, V, V, V, F, V, Z, V]
    lib.mla_decode.restype = I
    lib.mla_decode_f32.argtypes = [V, V, I, V, I, V, I, I, I, V, V, V, F, V, Z, V]
    lib.mla_decode_f32.restype = I
    lib.mla_decode_sparse_f32.argtypes = [V, V, I, V, I, V, V, I, V, I, I, V, V, V, F, V, Z, V]
    lib.mla_decode_sparse_f32.restype = I
    lib.mla_decode_attend.argtypes = [V, V, I, V, I, V, I, I, I, V, V, V, F, V, Z, V]
    lib.mla_decode_attend.restype = I
    lib.mla_decode_combine.argtypes = [I, I, I, V, V, V, V, Z, V]
    lib.mla_decode_combine.restype = I
    lib.mla_decode_noalloc.argtypes = [V, V, I, V, I, V, I, I, I, V, V, V, F, V]
    lib.mla_decode_noalloc.restype = I
    lib.mla_decode_sparse.argtypes = [V, V, I, V, I, V, V, I, V, I, I, V, V, V, F, V, Z, V]
    lib.mla_decode_sparse.restype = I
    lib.mla_cache_append.argtypes = [V, V, I, V, I, V, I, I, V]
    lib.mla_cache_append.restype = I
    lib.mla_q_absorb.argtypes = [V, V, V, V, I, I, I, V]
    lib.mla_q_absorb.restype = I
    lib.mla_gemm.argtypes = [V, V, V, I, I, I, I, I, V]
    lib.mla_gemm.restype = I
    lib.mla_attention_fwd.argtypes = [V, V, V, V, V, I, I, I, I, I, I, F, V]
    lib.mla_attention_fwd.restype = I
    lib.mla_selftest_wait_timeout.argtypes = [V]
    lib.mla_selftest_wait_timeout.restype = I
    lib.mla_check_device_error.argtypes = [V]
    lib.mla_check_device_error.restype = I
    lib.mla_strerror.argtypes = [I]
    lib.mla_strerror.restype = ctypes.c_char_p
    if path is None:
        _lib = lib
    return lib


def _ptr(x) -> int | None:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return int(x.data_ptr())


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        return int(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return stream
    return int(stream.cuda_stream)


def _check(rc: int, where: str) -> None:
    if rc != MLA_OK:
        raise MlaError(rc, where)


def mla_strerror(code: int) -> str:
    return load().mla_strerror(int(code)).decode()


def mla_num_clusters(device: int = 0) -> int:
    n = load().mla_num_clusters(int(device))
    _check(n if n < 0 else MLA_OK, "mla_num_clusters")
    return n


def mla_decode_kernel_kind(batch: int, s_q: int, h_q: int, max_pages: int, device: int = 0) -> int:
    """1 when mla_decode runs the narrow kernel for this shape, 0 for the
    general one."""
    k = load().mla_decode_kernel_kind(int(batch), int(s_q), int(h_q), int(max_pages), int(device))
    _check(k if k < 0 else MLA_OK, "mla_decode_kernel_kind")
    return k


def mla_plan_size(batch: int, s_q: int, h_q: int, device: int = 0) -> int:
    return int(load().mla_plan_size(batch, s_q, h_q, device))


def mla_plan_size_for_clusters(batch: int, s_q: int, h_q: int, num_clusters: int) -> int:
    return int(load().mla_plan_size_for_clusters(batch, s_q, h_q, num_clusters))


def mla_workspace_size(batch: int, s_q: int, h_q: int, device: int = 0) -> int:
    return int(load().mla_workspace_size(batch, s_q, h_q, device))


def mla_decode_plan(cache_seqlens, s_q: int, h_q: int, tile_meta, stream=None) -> None:
    """Device planner: cache_seqlens int32 [B] and tile_meta (bytes) on the GPU."""
    batch = int(cache_seqlens.shape[0])
    nbytes = int(tile_meta.numel() * tile_meta.element_size())
    rc = load().mla_decode_plan(_ptr(cache_seqlens), batch, s_q, h_q, _ptr(tile_meta), nbytes,
                                _stream(stream))
    _check(rc, "mla_decode_plan")


def mla_decode_plan_host(cache_seqlens, s_q: int, h_q: int, num_clusters: int) -> np.ndarray:
    """Host planner: returns the tile metadata as an int32 numpy array."""
    sl = np.ascontiguousarray(cache_seqlens, dtype=np.int32)
    batch = int(sl.shape[0])
    nbytes = mla_plan_size_for_clusters(batch, s_q, h_q, num_clusters)
    if nbytes == 0:
        raise MlaError(MLA_ERR_INVALID_ARG, "mla_plan_size_for_clusters")
    meta = np.zeros((nbytes + 7) // 8 * 2, dtype=np.int32)
    rc = load().mla_decode_plan_host(sl.ctypes.data, batch, s_q, h_q, num_clusters,
                                     meta.ctypes.data, meta.nbytes)
    _check(rc, "mla_decode_plan_host")
    return meta


def _decode(fn: str, q, kv_cache, block_table, cache_seqlens, tile_meta, out, lse,
            softmax_scale: float, workspace, stream) -> None:
    B, s_q, h_q = int(q.shape[0]), int(q.shape[1]), int(q.shape[2])
    rc = getattr(load(), fn)(_ptr(q), _ptr(kv_cache), int(kv_cache.shape[0]), _ptr(block_table),
                             int(block_table.shape[1]), _ptr(cache_seqlens), B, s_q, h_q,
                             _ptr(tile_meta), _ptr(out), _ptr(lse), float(softmax_scale),
                             _ptr(workspace), int(workspace.numel() * workspace.element_size()),
                             _stream(stream))
    _check(rc, fn)


def mla_decode(q, kv_cache, block_table, cache_seqlens, tile_meta, out, lse,
               softmax_scale: float, workspace, stream=None) -> None:
    """Decode attention on the GPU.

    q [B, s_q, h_q, 576] bf16; kv_cache [pages, 64, 1, 576] bf16; block_table
    [B, max_pages] int32; cache_seqlens [B] int32; out [B, s_q, h_q, 512] bf16;
    lse [B, h_q, s_q] fp32; tile_meta from mla_decode_plan; workspace of at
    least mla_workspace_size bytes.
    """
    _decode("mla_decode", q, kv_cache, block_table, cache_seqlens, tile_meta, out, lse,
            softmax_scale, workspace, stream)


def mla_decode_f32(q, kv_cache, block_table, cache_seqlens, tile_meta, out, lse,
                   softmax_scale: float, workspace, stream=None) -> None:
    """mla_decode with out fp32 [B, s_q, h_q, 512] (the unrounded result)."""
    _decode("mla_decode_f32", q, kv_cache, block_table, cache_seqlens, tile_meta, out, lse,
            softmax_scale, workspace, stream)


def _decode_sparse(fn: str, q, kv_cache, block_table, cache_seqlens, indices, counts, tile_meta,
                   out, lse, softmax_scale: float, workspace, stream) -> None:
    B, h_q = int(q.shape[0]), int(q.shape[2])
    if int(q.shape[1]) != 1:
        raise MlaError(MLA_ERR_INVALID_ARG, f"{fn} (s_q must be 1)")
    rc = getattr(load(), fn)(_ptr(q), _ptr(kv_cache), int(kv_cache.shape[0]),
                             _ptr(block_table), int(block_table.shape[1]),
                             _ptr(cache_seqlens), _ptr(indices), int(indices.shape[1]),
                             _ptr(counts), B, h_q, _ptr(tile_meta), _ptr(out), _ptr(lse),
                             float(softmax_scale), _ptr(workspace),
                             int(workspace.numel() * workspace.element_size()),
                             _stream(stream))
    _check(rc, fn)


def mla_decode_sparse(q, kv_cache, block_table, cache_seqlens, indices, counts, tile_meta, out,
                      lse, softmax_scale: float, workspace, stream=None) -> None:
    """Sparse decode: q [B, 1, h_q, 576]; indices [B, topk] int32 token
    positions; counts [B] int32; tile_meta from mla_decode_plan(counts, 1,
    h_q, ...); out [B, 1, h_q, 512] bf16; lse [B, h_q, 1] fp32."""
    _decode_sparse("mla_decode_sparse", q, kv_cache, block_table, cache_seqlens, indices, counts,
                   tile_meta, out, lse, softmax_scale, workspace, stream)


def mla_decode_sparse_f32(q, kv_cache, block_table, cache_seqlens, indices, counts, tile_meta,
                          out, lse, softmax_scale: float, workspace, stream=None) -> None:
    """mla_decode_sparse with out fp32 [B, 1, h_q, 512]."""
    _decode_sparse("mla_decode_sparse_f32", q, kv_cache, block_table, cache_seqlens, indices,
                   counts, tile_meta, out, lse, softmax_scale, workspace, stream)


def mla_decode_attend(q, kv_cache, block_table, cache_seqlens, tile_meta, out, lse,
                      softmax_scale: float, workspace, stream=None) -> None:
    """Main kernel only (see mla_decode_combine for the second half)."""
    B, s_q, h_q = int(q.shape[0]), int(q.shape[1]), int(q.shape[2])
    rc = load().mla_decode_attend(_ptr(q), _ptr(kv_cache), int(kv_cache.shape[0]),
                                  _ptr(block_table), int(block_table.shape[1]),
                                  _ptr(cache_seqlens), B, s_q, h_q, _ptr(tile_meta), _ptr(out),
                                  _ptr(lse), float(softmax_scale), _ptr(workspace),
                                  int(workspace.numel() * workspace.element_size()),
                                  _stream(stream))
    _check(rc, "mla_decode_attend")


def mla_decode_combine(batch: int, s_q: int, h_q: int, tile_meta, out, lse, workspace,
                       stream=None) -> None:
    """LSE-combine kernel only: merges the split partials left by the attend."""
    rc = load().mla_decode_combine(batch, s_q, h_q, _ptr(tile_meta), _ptr(out), _ptr(lse),
                                   _ptr(workspace),
                                   int(workspace.numel() * workspace.element_size()),
                                   _stream(stream))
    _check(rc, "mla_decode_combine")


def mla_decode_noalloc(q, kv_cache, block_table, cache_seqlens, tile_meta, out, lse,
                       softmax_scale: float, stream=None) -> None:
    """mla_decode without a workspace argument, for callers that cannot
    allocate device memory: the library's own static scratch holds the split
    partials (shared by all calls, so calls must not overlap on the GPU)."""
    B, s_q, h_q = int(q.shape[0]), int(q.shape[1]), int(q.shape[2])
    rc = load().mla_decode_noalloc(_ptr(q), _ptr(kv_cache), int(kv_cache.shape[0]),
                                   _ptr(block_table), int(block_table.shape[1]),
                                   _ptr(cache_seqlens), B, s_q, h_q, _ptr(tile_meta), _ptr(out),
                                   _ptr(lse), float(softmax_scale), _stream(stream))
    _check(rc, "mla_decode_noalloc")


def mla_selftest_wait_timeout(stream=None) -> None:
    """Failure-path self-test: a wait that nothing satisfies gives up after
    about 2 s and records MLA_ERR_DEVICE_TIMEOUT (see mla_check_device_error)."""
    _check(load().mla_selftest_wait_timeout(_stream(stream)), "mla_selftest_wait_timeout")


def mla_check_device_error(stream=None) -> int:
    return int(load().mla_check_device_error(_stream(stream)))


def mla_cache_append(kv_new, kv_cache, block_table, cache_seqlens, stream=None) -> None:
    """kv_new [B, s_q, 576] bf16 rows of the new tokens into kv_cache [pages,
    64, 1, 576] at positions cache_seqlens[b] - s_q + i (the lengths count
    the new tokens)."""
    B, s_q = int(kv_new.shape[0]), int(kv_new.shape[1])
    rc = load().mla_cache_append(_ptr(kv_new), _ptr(kv_cache), int(kv_cache.shape[0]),
                                 _ptr(block_table), int(block_table.shape[1]),
                                 _ptr(cache_seqlens), B, s_q, _stream(stream))
    _check(rc, "mla_cache_append")


def mla_q_absorb(q_nope, q_rope, w_uk, q, stream=None) -> None:
    """q [B, s_q, h_q, 576] bf16 = [q_nope W_UK per head | q_rope]; q_nope [B,
    s_q, h_q, 128], q_rope [B, s_q, h_q, 64], w_uk [h_q, 128, 512], all bf16."""
    B, s_q, h_q = int(q_nope.shape[0]), int(q_nope.shape[1]), int(q_nope.shape[2])
    rc = load().mla_q_absorb(_ptr(q_nope), _ptr(q_rope), _ptr(w_uk), _ptr(q), B, s_q, h_q,
                             _stream(stream))
    _check(rc, "mla_q_absorb")


def _dtype_code(t) -> int:
    import torch
    return {torch.float16: MLA_DTYPE_F16, torch.bfloat16: MLA_DTYPE_BF16,
            torch.float32: MLA_DTYPE_F32}[t.dtype]


def mla_gemm(a, b, c, stream=None) -> None:
    """c [M, N] = a [M, K] @ b [K, N] on the tensor cores (a, b fp16 or bf16
    of one type; c fp16, bf16 or fp32)."""
    M, K = int(a.shape[0]), int(a.shape[1])
    N = int(b.shape[1])
    rc = load().mla_gemm(_ptr(a), _ptr(b), _ptr(c), M, N, K, _dtype_code(a), _dtype_code(c),
                         _stream(stream))
    _check(rc, "mla_gemm")


def mla_attention_fwd(q, k, v, out, lse, causal: bool, softmax_scale: float,
                      stream=None) -> None:
    """Dense attention forward: q, k [B, S, H, d_qk], v [B, S, H, d_v], out
    [B, S, H, d_v] (bf16), lse [B, H, S] fp32."""
    B, S, H, dqk = (int(x) for x in q.shape)
    dv = int(v.shape[3])
    rc = load().mla_attention_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, S, H, dqk,
                                  dv, 1 if causal else 0, float(softmax_scale), _stream(stream))
    _check(rc, "mla_attention_fwd")


def alloc_plan_and_workspace(batch: int, s_q: int, h_q: int, device: int = 0):
    """torch buffers for the tile metadata and the split scratch."""
    import torch
    pbytes = mla_plan_size(batch, s_q, h_q, device)
    wbytes = mla_workspace_size(batch, s_q, h_q, device)
    if pbytes == 0 or wbytes == 0:
        raise MlaError(mla_num_clusters(device) if pbytes == 0 else MLA_ERR_INVALID_ARG,
                       "mla_plan_size/mla_workspace_size")
    dev = torch.device("cuda", device)
    tile_meta = torch.empty((pbytes + 7) // 8 * 2, dtype=torch.int32, device=dev)
    workspace = torch.empty(wbytes // 4 + 64, dtype=torch.float32, device=dev)
    return tile_meta, workspace
