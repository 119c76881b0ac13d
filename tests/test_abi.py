"""The C ABI loads, exports every declared symbol, and rejects bad arguments
on the host before touching a GPU (CPU only)."""
import ctypes
import os
import re

import pytest

from mla_decode_attention_07_gb300 import libmla

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build_library()
    return libmla.load()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "mla.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mla_\w+)\s*\(", text)))


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert names and set(names) == set(libmla.EXPORTED)
    for n in names:
        assert hasattr(lib, n), n


def test_strerror(lib):
    for code in range(0, -8, -1):
        s = libmla.mla_strerror(code)
        assert s and s != "unknown error"
    assert libmla.mla_strerror(-99) == "unknown error"


def _decode(lib, **kw):
    a = dict(q=0x1000, kv=0x2000, num_pages=4, bt=0x3000, max_pages=4, sl=0x4000, batch=1, s_q=1,
             h_q=16, meta=0x5000, out=0x6000, lse=0x7000, scale=0.07, ws=0x8000,
             ws_bytes=1 << 30, stream=None)
    a.update(kw)
    return lib.mla_decode(a["q"], a["kv"], a["num_pages"], a["bt"], a["max_pages"], a["sl"],
                          a["batch"], a["s_q"], a["h_q"], a["meta"], a["out"], a["lse"],
                          ctypes.c_float(a["scale"]), a["ws"], a["ws_bytes"], a["stream"])


@pytest.mark.parametrize("kw", [
    dict(q=None), dict(kv=None), dict(bt=None), dict(sl=None), dict(meta=None), dict(out=None),
    dict(lse=None), dict(batch=0), dict(s_q=0), dict(s_q=9), dict(h_q=0), dict(h_q=129),
    dict(num_pages=0), dict(max_pages=0), dict(num_pages=1 << 25), dict(q=0x1008),
    dict(kv=0x2004), dict(out=0x6002), dict(lse=0x7002), dict(scale=float("nan")),
])
def test_decode_rejects_bad_args_on_host(lib, kw):
    assert _decode(lib, **kw) == libmla.MLA_ERR_INVALID_ARG


def _sparse(lib, **kw):
    a = dict(q=0x1000, kv=0x2000, num_pages=4, bt=0x3000, max_pages=4, sl=0x4000, idx=0x9000,
             topk=64, cnt=0xA000, batch=1, h_q=16, meta=0x5000, out=0x6000, lse=0x7000,
             scale=0.07, ws=0x8000, ws_bytes=1 << 30, stream=None)
    a.update(kw)
    return lib.mla_decode_sparse(a["q"], a["kv"], a["num_pages"], a["bt"], a["max_pages"],
                                 a["sl"], a["idx"], a["topk"], a["cnt"], a["batch"], a["h_q"],
                                 a["meta"], a["out"], a["lse"], ctypes.c_float(a["scale"]),
                                 a["ws"], a["ws_bytes"], a["stream"])


@pytest.mark.parametrize("kw", [
    dict(idx=None), dict(cnt=None), dict(sl=None), dict(topk=0), dict(idx=0x9002),
    dict(cnt=0xA001), dict(batch=1 << 16, topk=1 << 16), dict(q=None), dict(h_q=0),
    dict(out=0x6002), dict(scale=float("inf")),
])
def test_sparse_rejects_bad_args_on_host(lib, kw):
    assert _sparse(lib, **kw) == libmla.MLA_ERR_INVALID_ARG


@pytest.mark.parametrize("args", [
    (None, 0x2000, 0x3000, 64, 64, 64), (0x1000, None, 0x3000, 64, 64, 64),
    (0x1000, 0x2000, None, 64, 64, 64), (0x1000, 0x2000, 0x3000, 0, 64, 64),
    (0x1000, 0x2000, 0x3000, 64, 60, 64), (0x1000, 0x2000, 0x3000, 64, 64, 12),
    (0x1008, 0x2000, 0x3000, 64, 64, 64), (0x1000, 0x2000, 0x3004, 64, 64, 64),
])
def test_gemm_rejects_bad_args_on_host(lib, args):
    A, B, C, M, N, K = args
    assert lib.mla_gemm(A, B, C, M, N, K, 0, 0, None) == libmla.MLA_ERR_INVALID_ARG
    assert lib.mla_gemm(0x1000, 0x2000, 0x3000, 64, 64, 64, 2, 0, None) == \
        libmla.MLA_ERR_INVALID_ARG                         # fp32 inputs are not supported
    assert lib.mla_gemm(0x1000, 0x2000, 0x3000, 64, 64, 64, 0, 3, None) == \
        libmla.MLA_ERR_INVALID_ARG


def test_prologue_rejects_bad_args_on_host(lib):
    E = libmla.MLA_ERR_INVALID_ARG
    assert lib.mla_q_absorb(None, 0x2000, 0x3000, 0x4000, 1, 1, 16, None) == E
    assert lib.mla_q_absorb(0x1000, 0x2008, 0x3000, 0x4000, 1, 1, 16, None) == E
    assert lib.mla_q_absorb(0x1000, 0x2000, 0x3000, 0x4000, 1, 0, 16, None) == E
    assert lib.mla_cache_append(0x1000, 0x2000, 4, 0x3000, 4, 0x4000, 0, 1, None) == E
    assert lib.mla_cache_append(0x1000, 0x2000, 4, 0x3002, 4, 0x4000, 1, 1, None) == E
    assert lib.mla_cache_append(0x1004, 0x2000, 4, 0x3000, 4, 0x4000, 1, 1, None) == E
    assert lib.mla_cache_append(0x1000, 0x2000, 0, 0x3000, 4, 0x4000, 1, 1, None) == E


@pytest.mark.parametrize("kw", [
    dict(q=None), dict(lse=None), dict(batch=0), dict(seqlen=0), dict(heads=0), dict(dqk=96),
    dict(dqk=256), dict(dv=64), dict(scale=0.0), dict(scale=float("nan")), dict(out=0x4008),
    dict(lse=0x5002),
])
def test_attention_rejects_bad_args_on_host(lib, kw):
    a = dict(q=0x1000, k=0x2000, v=0x3000, out=0x4000, lse=0x5000, batch=1, seqlen=128,
             heads=2, dqk=128, dv=128, causal=1, scale=0.08)
    a.update(kw)
    rc = lib.mla_attention_fwd(a["q"], a["k"], a["v"], a["out"], a["lse"], a["batch"],
                               a["seqlen"], a["heads"], a["dqk"], a["dv"], a["causal"],
                               ctypes.c_float(a["scale"]), None)
    assert rc == libmla.MLA_ERR_INVALID_ARG


def test_plan_rejects_bad_args_on_host(lib):
    assert lib.mla_decode_plan(None, 1, 1, 16, 0x5000, 4096, None) == libmla.MLA_ERR_INVALID_ARG
    assert lib.mla_decode_plan(0x4000, 1, 1, 0, 0x5000, 4096, None) == libmla.MLA_ERR_INVALID_ARG
    assert lib.mla_decode_plan(0x4000, 1, 1, 16, 0x5004, 4096, None) == libmla.MLA_ERR_INVALID_ARG


def test_plan_host_checks_buffer_size(lib):
    import numpy as np
    sl = np.array([100], dtype=np.int32)
    meta = np.zeros(4, dtype=np.int64)
    rc = lib.mla_decode_plan_host(sl.ctypes.data, 1, 1, 16, 8, meta.ctypes.data, meta.nbytes)
    assert rc == libmla.MLA_ERR_WORKSPACE


def test_no_gpu_means_error_not_fallback(lib):
    from conftest import gpu_available
    if gpu_available():
        pytest.skip("a GPU is present")
    # Valid-looking arguments: the only thing missing is the device.
    assert _decode(lib) in (libmla.MLA_ERR_CUDA, libmla.MLA_ERR_UNSUPPORTED_DEVICE)
    assert _sparse(lib) in (libmla.MLA_ERR_CUDA, libmla.MLA_ERR_UNSUPPORTED_DEVICE)
    assert lib.mla_num_clusters(0) < 0
    assert lib.mla_plan_size(1, 1, 16, 0) == 0
    assert lib.mla_gemm(0x1000, 0x2000, 0x3000, 64, 64, 64, 0, 0, None) in \
        (libmla.MLA_ERR_CUDA, libmla.MLA_ERR_UNSUPPORTED_DEVICE)
    assert lib.mla_cache_append(0x1000, 0x2000, 4, 0x3000, 4, 0x4000, 1, 1, None) in \
        (libmla.MLA_ERR_CUDA, libmla.MLA_ERR_UNSUPPORTED_DEVICE)


@pytest.mark.parametrize("args", [(0, 1, 16, 4), (1, 0, 16, 4), (1, 9, 16, 4), (1, 1, 0, 4),
                                  (1, 1, 129, 4), (1, 1, 16, 0)])
def test_kernel_kind_rejects_bad_shapes_on_host(lib, args):
    assert lib.mla_decode_kernel_kind(*args, 0) == libmla.MLA_ERR_INVALID_ARG
