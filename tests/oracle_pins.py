"""Checks that pin the fp64 oracle to facts that do not come from the oracle.

Each ``check_*`` takes an ``oracle.Oracle`` and raises AssertionError when the
oracle disagrees with the fact it checks.  They are collected by
``test_oracle_pins.py`` (against the real oracle) and by
``test_oracle_mutants.py`` (against copies of the oracle with a planted
mistake, each of which at least one check must reject).

What pins what:
  dense          - paging, gather, causal offset: a dense numpy evaluation of
                   softmax(Q K^T * scale) V over the explicitly gathered rows
  seqlen_one     - one visible key: out is that key's first 512 dims, lse is
                   scale * q.k (exact fp64 dot of bf16 values via math.fsum)
  constant_v     - softmax weights sum to one: equal value rows come back
  shift          - a logit shift common to all keys leaves out alone and moves
                   lse by exactly that shift
  q_zero         - closed form: out = mean of visible value rows, lse = ln n
  split_combine  - attention over disjoint key ranges merged through lse
                   equals attention over their union
  causal         - token 0 of a two-token query equals a one-token query
                   over L - 1 keys; token 1 equals one over L keys
  permutation    - relabelling the pool pages (and the block table with them)
                   changes nothing, bit for bit
  two_token      - closed form with two keys, hand-chosen exact values
  empty          - no visible key: out = 0, lse = -inf
  sparse_dense   - sparse decode: a dense numpy evaluation over the rows at
                   the listed token positions (distinct, repeated, partial
                   counts, and the identity list, which is the dense case)
  sparse_twice   - every position listed twice: out unchanged, lse + ln 2
  sparse_order   - the order of the list does not matter
  sparse_edges   - count 0 gives out = 0, lse = -inf; a position past L_b
                   is rejected
"""
from __future__ import annotations

import math

import numpy as np

from mla_decode_attention_07_gb300 import workloads as W

SCALE = W.SOFTMAX_SCALE


def bf(x):
    a = np.asarray(x, dtype=np.float32)
    return W.float32_to_bf16_bits(a).reshape(a.shape)


def f64(bits):
    return W.bf16_bits_to_float32(bits).astype(np.float64)


def dense_reference(inp):
    """softmax(Q K^T * scale) V evaluated densely with numpy matmuls."""
    B, s_q, h_q = inp.batch, inp.s_q, inp.h_q
    out = np.zeros((B, s_q, h_q, W.D_V))
    lse = np.zeros((B, h_q, s_q))
    for b in range(B):
        L = int(inp.cache_seqlens[b])
        rows = [inp.kv_cache[inp.block_table[b, t // W.PAGE], t % W.PAGE, 0] for t in range(L)]
        K = f64(np.stack(rows)) if rows else np.zeros((0, W.D_QK))
        for i in range(s_q):
            n = L - s_q + 1 + i
            if n <= 0:
                lse[b, :, i] = -np.inf
                continue
            Q = f64(inp.q[b, i])                    # [h, 576]
            S = (Q @ K[:n].T) * inp.softmax_scale   # [h, n]
            m = S.max(axis=1, keepdims=True)
            P = np.exp(S - m)
            l = P.sum(axis=1)
            out[b, i] = (P @ K[:n, : W.D_V]) / l[:, None]
            lse[b, :, i] = m[:, 0] + np.log(l)
    return out, lse


def _close(a, b, tol, what):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    assert a.shape == b.shape, f"{what}: shape {a.shape} vs {b.shape}"
    same_inf = (np.isinf(a) & np.isinf(b) & (np.sign(a) == np.sign(b)))
    diff = np.where(same_inf, 0.0, np.abs(a - b))
    assert np.all(np.isfinite(diff)), f"{what}: non-finite mismatch"
    err = float(diff.max()) if diff.size else 0.0
    assert err <= tol, f"{what}: max |err| {err:.3e} > {tol:.1e}"


def check_dense(orc):
    cases = [
        dict(seed=11, batch=2, s_q=1, h_q=4, seqlens=[1, 130], extra_pages=2),
        dict(seed=12, batch=3, s_q=2, h_q=3, seqlens=[2, 64, 65], extra_pages=1),
        dict(seed=13, batch=1, s_q=1, h_q=16, seqlens=[256], extra_pages=0),
        dict(seed=14, batch=2, s_q=2, h_q=2, seqlens=[129, 7], extra_pages=3),
    ]
    for c in cases:
        inp = W.make_inputs(c["seed"], c["batch"], c["s_q"], c["h_q"], c["seqlens"],
                            extra_pages=c["extra_pages"])
        o, l = orc.mla_decode(inp, nthreads=2)
        ro, rl = dense_reference(inp)
        _close(o, ro, 1e-12, f"dense out {c}")
        _close(l, rl, 1e-12, f"dense lse {c}")


def check_seqlen_one(orc):
    inp = W.make_inputs(21, 2, 1, 3, [1, 1])
    o, l = orc.mla_decode(inp, nthreads=1)
    for b in range(2):
        k = inp.kv_cache[inp.block_table[b, 0], 0, 0]
        for h in range(3):
            _close(o[b, 0, h], f64(k[: W.D_V]), 0.0, "seqlen=1 out")
            dot = math.fsum(float(x) * float(y) for x, y in zip(f64(inp.q[b, 0, h]), f64(k)))
            _close(l[b, h, 0], SCALE * dot, 1e-12, "seqlen=1 lse")


def check_constant_v(orc):
    inp = W.make_inputs(22, 2, 2, 4, [150, 65])
    row = bf(np.linspace(-3.0, 3.0, W.D_V))
    for b in range(2):
        L = int(inp.cache_seqlens[b])
        for t in range(L):
            inp.kv_cache[inp.block_table[b, t // W.PAGE], t % W.PAGE, 0, : W.D_V] = row
    o, _ = orc.mla_decode(inp, nthreads=2)
    want = np.broadcast_to(f64(row), o.shape)
    _close(o, want, 1e-12, "constant V")


def check_shift(orc):
    base = W.make_inputs(23, 2, 2, 3, [200, 70])
    d = W.D_QK - 1
    for b in range(2):
        L = int(base.cache_seqlens[b])
        for t in range(L):
            base.kv_cache[base.block_table[b, t // W.PAGE], t % W.PAGE, 0, d] = bf(2.0)
    base.q[..., d] = bf(0.0)
    o0, l0 = orc.mla_decode(base, nthreads=2)
    base.q[..., d] = bf(0.5)
    o1, l1 = orc.mla_decode(base, nthreads=2)
    _close(o1, o0, 1e-12, "shift out")
    _close(l1 - l0, np.full_like(l0, SCALE * 1.0), 1e-12, "shift lse")


def check_q_zero(orc):
    inp = W.make_inputs(24, 3, 2, 2, [1, 77, 130], q_zero=True)
    o, l = orc.mla_decode(inp, nthreads=2)
    for b in range(3):
        L = int(inp.cache_seqlens[b])
        for i in range(2):
            n = L - 2 + 1 + i
            if n <= 0:
                _close(o[b, i], np.zeros_like(o[b, i]), 0.0, "q=0 empty out")
                assert np.all(np.isneginf(l[b, :, i])), "q=0 empty lse"
                continue
            V = f64(np.stack([inp.kv_cache[inp.block_table[b, t // W.PAGE], t % W.PAGE, 0, : W.D_V]
                              for t in range(n)]))
            _close(o[b, i], np.broadcast_to(V.mean(axis=0), o[b, i].shape), 1e-12, "q=0 out")
            _close(l[b, :, i], np.full(2, math.log(n)), 1e-12, "q=0 lse")


def check_split_combine(orc):
    inp = W.make_inputs(25, 1, 2, 4, [300])
    rows = [(0, i, h) for i in range(2) for h in range(4)]
    full_o, full_l = orc.mla_decode_rows(inp, rows, nthreads=2)
    for cuts in [(0, 64), (64, 128), (100, 101), (1, 299), (150, 400)]:
        a, b = cuts
        parts = [orc.mla_decode_rows(inp, rows, 0, a, nthreads=2),
                 orc.mla_decode_rows(inp, rows, a, b, nthreads=2),
                 orc.mla_decode_rows(inp, rows, b, 2**31 - 1, nthreads=2)]
        for r in range(len(rows)):
            lse, out = orc.lse_combine([p[1][r] for p in parts], [p[0][r] for p in parts])
            _close(out, full_o[r], 1e-12, f"split {cuts} out")
            _close(lse, full_l[r], 1e-12, f"split {cuts} lse")


def check_causal(orc):
    two = W.make_inputs(26, 2, 2, 3, [90, 64])
    for i, delta in ((0, 1), (1, 0)):
        one = W.DecodeInputs(q=np.ascontiguousarray(two.q[:, i:i + 1]), kv_cache=two.kv_cache,
                             block_table=two.block_table,
                             cache_seqlens=(two.cache_seqlens - delta).astype(np.int32),
                             s_q=1, h_q=3)
        o2, l2 = orc.mla_decode(two, nthreads=2)
        o1, l1 = orc.mla_decode(one, nthreads=2)
        _close(o2[:, i], o1[:, 0], 1e-12, f"causal token {i} out")
        _close(l2[:, :, i], l1[:, :, 0], 1e-12, f"causal token {i} lse")


def check_permutation(orc):
    inp = W.make_inputs(27, 3, 1, 2, [65, 1, 200], extra_pages=2)
    o0, l0 = orc.mla_decode(inp, nthreads=2)
    relabel = W.permutation(99, 1, inp.num_pages)
    kv = np.empty_like(inp.kv_cache)
    kv[relabel] = inp.kv_cache
    moved = W.DecodeInputs(q=inp.q, kv_cache=kv, block_table=relabel[inp.block_table],
                           cache_seqlens=inp.cache_seqlens, s_q=1, h_q=2)
    o1, l1 = orc.mla_decode(moved, nthreads=2)
    assert np.array_equal(o0, o1) and np.array_equal(l0, l1), "page relabelling changed result"


def check_two_token(orc):
    inp = W.make_inputs(28, 1, 1, 1, [2], poison=False)
    page = inp.block_table[0, 0]
    inp.q[:] = bf(0.0)
    inp.q[0, 0, 0, 0] = bf(1.0)
    inp.kv_cache[page, :2] = bf(0.0)
    k0 = inp.kv_cache[page, 0, 0]
    k1 = inp.kv_cache[page, 1, 0]
    k0[1] = bf(1.0)
    k0[100] = bf(7.0)
    k0[520] = bf(5.0)          # rope dim: never part of the values
    k1[0] = bf(4.0)
    k1[1] = bf(-2.0)
    k1[2] = bf(0.5)
    o, l = orc.mla_decode(inp, nthreads=1)
    s1 = SCALE * 4.0
    lse = math.log(1.0 + math.exp(s1))
    w0, w1 = math.exp(-lse), math.exp(s1 - lse)
    want = np.zeros(W.D_V)
    want[0] = 4.0 * w1
    want[1] = 1.0 * w0 - 2.0 * w1
    want[2] = 0.5 * w1
    want[100] = 7.0 * w0
    _close(o[0, 0, 0], want, 1e-14, "two-token out")
    _close(l[0, 0, 0], lse, 1e-14, "two-token lse")


def check_empty(orc):
    inp = W.make_inputs(29, 3, 2, 2, [0, 1, 3])
    o, l = orc.mla_decode(inp, nthreads=1)
    assert np.all(o[0] == 0.0) and np.all(np.isneginf(l[0])), "L=0 row not empty"
    assert np.all(o[1, 0] == 0.0) and np.all(np.isneginf(l[1, :, 0])), "L=1 token 0 not empty"
    k = inp.kv_cache[inp.block_table[1, 0], 0, 0]
    _close(o[1, 1], np.broadcast_to(f64(k[: W.D_V]), o[1, 1].shape), 0.0, "L=1 token 1")
    assert np.all(np.isfinite(l[2])), "L=3 rows finite"


def _sparse(orc, si, nthreads=2):
    """The oracle on valid sparse inputs; refusing them is a failed pin."""
    try:
        return orc.mla_decode_sparse(si, nthreads=nthreads)
    except ValueError as e:
        raise AssertionError(f"oracle rejected valid sparse inputs: {e}") from e


def sparse_reference(si):
    """softmax(q K_sel^T * scale) V_sel per (b, h), K_sel the cache rows at
    the listed positions, evaluated with numpy matmuls."""
    inp = si.base
    B, h_q = inp.batch, inp.h_q
    out = np.zeros((B, 1, h_q, W.D_V))
    lse = np.zeros((B, h_q, 1))
    for b in range(B):
        c = int(si.counts[b])
        if c == 0:
            lse[b] = -np.inf
            continue
        ts = [int(t) for t in si.indices[b, :c]]
        K = f64(np.stack([inp.kv_cache[inp.block_table[b, t // W.PAGE], t % W.PAGE, 0] for t in ts]))
        S = (f64(inp.q[b, 0]) @ K.T) * inp.softmax_scale
        m = S.max(axis=1, keepdims=True)
        P = np.exp(S - m)
        l = P.sum(axis=1)
        out[b, 0] = (P @ K[:, : W.D_V]) / l[:, None]
        lse[b, :, 0] = m[:, 0] + np.log(l)
    return out, lse


def check_sparse_dense(orc):
    cases = [
        dict(seed=31, seqlens=[300, 64, 1], topk=128, counts=None, repeats=False),
        dict(seed=32, seqlens=[500, 200], topk=70, counts=[70, 13], repeats=False),
        dict(seed=33, seqlens=[90, 40], topk=64, counts=[64, 30], repeats=True),
    ]
    for c in cases:
        si = W.make_sparse_inputs(c["seed"], len(c["seqlens"]), 3, c["seqlens"], c["topk"],
                                  c["counts"], repeats=c["repeats"])
        o, l = _sparse(orc, si)
        ro, rl = sparse_reference(si)
        _close(o, ro, 1e-12, f"sparse out {c}")
        _close(l, rl, 1e-12, f"sparse lse {c}")
    # the identity list over the whole sequence is the dense case
    inp = W.make_inputs(34, 2, 1, 2, [130, 65], extra_pages=1)
    idx = np.full((2, 130), -1, dtype=np.int32)
    idx[0, :130] = np.arange(130)
    idx[1, :65] = np.arange(65)
    si = W.SparseInputs(base=inp, indices=idx, counts=np.array([130, 65], dtype=np.int32))
    o, l = _sparse(orc, si)
    ro, rl = dense_reference(inp)
    _close(o, ro, 1e-12, "sparse identity out")
    _close(l, rl, 1e-12, "sparse identity lse")


def check_sparse_twice(orc):
    si = W.make_sparse_inputs(35, 2, 2, [200, 77], 40)
    o1, l1 = _sparse(orc, si)
    idx2 = np.concatenate([si.indices[:, :40], si.indices[:, :40]], axis=1)
    two = W.SparseInputs(base=si.base, indices=idx2, counts=(2 * si.counts).astype(np.int32))
    o2, l2 = _sparse(orc, two)
    _close(o2, o1, 1e-12, "listed twice out")
    _close(l2 - l1, np.full_like(l1, math.log(2.0)), 1e-12, "listed twice lse")


def check_sparse_order(orc):
    si = W.make_sparse_inputs(36, 2, 3, [256, 100], 64)
    o1, l1 = _sparse(orc, si)
    idx = si.indices.copy()
    for b in range(2):
        c = int(si.counts[b])
        idx[b, :c] = idx[b, :c][W.permutation(37 + b, 1, c)]
    o2, l2 = _sparse(orc, W.SparseInputs(base=si.base, indices=idx, counts=si.counts))
    assert not np.array_equal(idx, si.indices), "order check did not reorder"
    _close(o2, o1, 1e-12, "reordered out")
    _close(l2, l1, 1e-12, "reordered lse")


def check_sparse_edges(orc):
    si = W.make_sparse_inputs(38, 2, 2, [100, 50], 16, counts=[0, 16])
    o, l = _sparse(orc, si, nthreads=1)
    assert np.all(o[0] == 0.0) and np.all(np.isneginf(l[0])), "count 0 not empty"
    assert np.all(np.isfinite(l[1])), "count 16 finite"
    bad = si.indices.copy()
    bad[1, 3] = 50                              # == L_1: past the sequence
    try:
        orc.mla_decode_sparse(W.SparseInputs(base=si.base, indices=bad, counts=si.counts),
                              nthreads=1)
    except ValueError:
        pass
    else:
        raise AssertionError("a position past L_b was accepted")


ALL_CHECKS = [check_dense, check_seqlen_one, check_constant_v, check_shift, check_q_zero,
              check_split_combine, check_causal, check_permutation, check_two_token,
              check_empty, check_sparse_dense, check_sparse_twice, check_sparse_order,
              check_sparse_edges]
