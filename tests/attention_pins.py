"""Pins of the dense attention oracle (attention_oracle.c).

Each check takes an ``oracle.Attention`` and raises AssertionError when the
oracle disagrees with something fixed independently of its code: a two-key
closed form, a single visible key, constant values, a common logit shift,
q = 0 (the mean of the visible rows), and the decode oracle (mla_oracle.c,
pinned on its own), which must agree row for row when the values are the
first 512 dims of 576-wide keys.
"""
import math

import numpy as np

import oracle as oracle_pkg
from mla_decode_attention_07_gb300 import workloads as W


def _f(bits):
    return W.bf16_bits_to_float32(bits).astype(np.float64)


def _bits(x):
    return W.float32_to_bf16_bits(np.asarray(x, dtype=np.float32))


def check_two_key_closed_form(orc):
    """scale 1, d_qk = d_v = 1, q = 1, keys 0 and 1, values 3 and -1:
    query 1 weighs them 1 / (1 + e) and e / (1 + e)."""
    q = _bits(np.ones((1, 2, 1, 1)))
    k = _bits(np.array([0.0, 1.0]).reshape(1, 2, 1, 1))
    v = _bits(np.array([3.0, -1.0]).reshape(1, 2, 1, 1))
    ai = W.AttentionInputs(q=q, k=k, v=v, causal=True, scale=1.0)
    out, lse = orc.attention(ai)
    e = math.e
    assert abs(out[0, 1, 0, 0] - (3.0 - e) / (1.0 + e)) < 1e-13
    assert abs(lse[0, 0, 1] - math.log(1.0 + e)) < 1e-13
    assert out[0, 0, 0, 0] == 3.0 and lse[0, 0, 0] == 0.0       # query 0 sees key 0 only


def check_first_row_and_single_key(orc):
    """Causal query 0 sees only key 0: out = v_0, lse = scale * q.k_0
    (summed exactly with math.fsum)."""
    ai = W.make_attention_inputs(41, 2, 50, 3, 64, 32)
    out, lse = orc.attention(ai)
    for b in range(2):
        for h in range(3):
            assert np.array_equal(out[b, 0, h], _f(ai.v[b, 0, h]))
            dot = math.fsum(float(x) for x in _f(ai.q[b, 0, h]) * _f(ai.k[b, 0, h]))
            assert abs(lse[b, h, 0] - ai.scale * dot) < 1e-12


def check_constant_values(orc):
    ai = W.make_attention_inputs(42, 1, 40, 2, 32, 16, causal=False)
    ai.v[...] = _bits(np.full((1, 40, 2, 16), 1.5))
    out, _ = orc.attention(ai)
    assert np.abs(out - 1.5).max() < 1e-13


def check_logit_shift(orc):
    """Key dim 0 set to 2 for every key; moving q's dim 0 by 0.5 shifts every
    logit of the row by scale, leaving out unchanged and lse + scale."""
    ai = W.make_attention_inputs(43, 1, 30, 2, 16, 8)
    ai.k[..., 0] = _bits(np.full((1, 30, 2), 2.0))
    ai.q[..., 0] = 0
    o0, l0 = orc.attention(ai)
    ai.q[..., 0] = _bits(np.full((1, 30, 2), 0.5))
    o1, l1 = orc.attention(ai)
    assert np.abs(o1 - o0).max() < 1e-12
    assert np.abs((l1 - l0) - ai.scale).max() < 1e-12


def check_zero_query(orc):
    """q = 0: every visible key weighs the same; causal row i is the mean of
    v_0..v_i and lse = ln(i + 1)."""
    ai = W.make_attention_inputs(44, 1, 20, 2, 16, 8)
    ai.q[...] = 0
    out, lse = orc.attention(ai)
    v = _f(ai.v)
    for i in (0, 7, 19):
        assert np.abs(out[0, i] - v[0, : i + 1].mean(axis=0)).max() < 1e-12
        assert np.abs(lse[0, :, i] - math.log(i + 1)).max() < 1e-12


def check_matches_decode_oracle(orc):
    """With d_qk = 576 and the values the first 512 dims of the keys, causal
    row i of one head is the MLA decode of a single query over the first i + 1
    cache rows: compare with the decode oracle through a paged cache whose
    pages are the keys in a shuffled order."""
    S, H = 130, 2
    ai = W.make_attention_inputs(45, 1, S, H, 576, 512)
    ai.v[...] = ai.k[..., :512]
    out, lse = orc.attention(ai)
    dec = oracle_pkg.Oracle(oracle_pkg.build())
    n_pages = 3
    perm = np.array([2, 0, 1], dtype=np.int32)
    for h in range(H):
        kv = np.zeros((n_pages, 64, 1, 576), dtype=np.uint16)
        for t in range(S):
            kv[perm[t // 64], t % 64, 0] = ai.k[0, t, h]
        for i in (0, 63, 64, 129):
            inp = W.DecodeInputs(q=ai.q[0, i, h].reshape(1, 1, 1, 576).copy(), kv_cache=kv,
                                 block_table=perm.reshape(1, 3),
                                 cache_seqlens=np.array([i + 1], dtype=np.int32), s_q=1, h_q=1,
                                 softmax_scale=ai.scale)
            ro, rl = dec.mla_decode(inp)
            assert np.abs(out[0, i, h] - ro[0, 0, 0]).max() < 1e-12
            assert abs(lse[0, h, i] - rl[0, 0, 0]) < 1e-12


def check_non_causal_last_row_and_rows_entry(orc):
    ai = W.make_attention_inputs(46, 2, 33, 2, 32, 16)
    oc, lc = orc.attention(ai)
    ai2 = W.AttentionInputs(q=ai.q, k=ai.k, v=ai.v, causal=False, scale=ai.scale)
    on, ln = orc.attention(ai2)
    assert np.array_equal(oc[:, -1], on[:, -1]) and np.array_equal(lc[..., -1], ln[..., -1])
    assert not np.allclose(oc[:, 0], on[:, 0])
    rows = np.array([[1, 0, 5], [0, 1, 32], [1, 1, 0]], dtype=np.int32)
    ro, rl = orc.attention_rows(ai, rows)
    for j, (b, h, i) in enumerate(rows):
        assert np.array_equal(ro[j], oc[b, i, h]) and rl[j] == lc[b, h, i]


ALL_CHECKS = [check_two_key_closed_form, check_first_row_and_single_key, check_constant_values,
              check_logit_shift, check_zero_query, check_matches_decode_oracle,
              check_non_causal_last_row_and_rows_entry]
