"""Pins of the cache-append and query-absorption oracle (prologue_oracle.c).

Each check takes an ``oracle.Prologue`` and raises AssertionError when the
oracle disagrees with something fixed independently of its code: slots
listed by hand, closed forms of the contraction (identity, one-hot, a 2 x 2
example worked by hand), linearity and head relabelling.  The mutant tests
run every check against copies of the oracle with one planted mistake.
"""
import numpy as np

from mla_decode_attention_07_gb300 import workloads as W

ROW = 576


def _bits(x):
    return W.float32_to_bf16_bits(np.asarray(x, dtype=np.float32))


def _cache(pages, seed=5):
    return W.normal_bf16(seed, 0x5A5A, pages * 64 * ROW).reshape(pages, 64, 1, ROW)


def check_append_hand_slots(orc):
    """Entry 0 has 65 tokens of which the last 2 are new: positions 63 and 64
    land in page 4 slot 63 and page 1 slot 0; entry 1 has 2 tokens, both new:
    page 2 slots 0 and 1.  Every other row is untouched."""
    cache = _cache(6)
    bt = np.array([[4, 1, -1], [2, 5, -1]], dtype=np.int32)
    sl = np.array([65, 2], dtype=np.int32)
    new = W.normal_bf16(6, 0x1234, 2 * 2 * ROW).reshape(2, 2, ROW)
    got = orc.cache_append(new, cache, bt, sl)
    expect = cache.copy()
    expect[4, 63, 0] = new[0, 0]
    expect[1, 0, 0] = new[0, 1]
    expect[2, 0, 0] = new[1, 0]
    expect[2, 1, 0] = new[1, 1]
    assert np.array_equal(got, expect)


def check_append_single_token(orc):
    """s_q = 1: length 1 writes slot 0 of the first page, length 128 slot 63
    of the second."""
    cache = _cache(4, seed=8)
    bt = np.array([[3, 0], [1, 2]], dtype=np.int32)
    sl = np.array([1, 128], dtype=np.int32)
    new = W.normal_bf16(9, 0x2222, 2 * ROW).reshape(2, 1, ROW)
    got = orc.cache_append(new, cache, bt, sl)
    expect = cache.copy()
    expect[3, 0, 0] = new[0, 0]
    expect[2, 63, 0] = new[1, 0]
    assert np.array_equal(got, expect)


def check_append_rejects_out_of_range(orc):
    """A sequence shorter than its new tokens, or a page index outside the
    pool, is an error; nothing is written."""
    cache = _cache(2, seed=3)
    new = W.normal_bf16(4, 0x3333, 2 * ROW).reshape(1, 2, ROW)
    for bt, sl in ((np.array([[0, 1]], np.int32), np.array([1], np.int32)),
                   (np.array([[0, 7]], np.int32), np.array([66], np.int32))):
        try:
            orc.cache_append(new, cache, bt, sl)
        except ValueError:
            continue
        raise AssertionError("out-of-range append accepted")


def check_append_then_gather(orc):
    """Reading the sequence back page by page through the block table (a
    walk written here, not the oracle's arithmetic) finds the new rows as its
    last s_q tokens."""
    rng = np.random.default_rng(11)
    pages = 9
    cache = _cache(pages, seed=12)
    bt = rng.permutation(pages).astype(np.int32).reshape(3, 3)
    sl = np.array([130, 64, 3], dtype=np.int32)
    s_q = 3
    new = W.normal_bf16(13, 0x4444, 3 * s_q * ROW).reshape(3, s_q, ROW)
    got = orc.cache_append(new, cache, bt, sl)
    for b in range(3):
        seq = np.concatenate([got[p, :, 0] for p in bt[b]])[: sl[b]]
        assert np.array_equal(seq[-s_q:], new[b])
        old = np.concatenate([cache[p, :, 0] for p in bt[b]])[: sl[b]]
        assert np.array_equal(seq[:-s_q], old[:-s_q])


def check_absorb_hand_example(orc):
    """Two heads, d_nope = d_c = 2, worked by hand:
    head 0: q = (1, 2), W = [[1, 0], [0.5, 2]] -> (1 + 1, 0 + 4) = (2, 4);
    head 1: q = (3, -1), W = [[2, 1], [1, 1]] -> (6 - 1, 3 - 1) = (5, 2)."""
    q = _bits([[[[1, 2], [3, -1]]]])
    w = _bits([[[1, 0], [0.5, 2]], [[2, 1], [1, 1]]])
    out = orc.q_absorb(q, w)
    assert np.array_equal(out[0, 0], np.array([[2.0, 4.0], [5.0, 2.0]]))


def check_absorb_identity(orc):
    """W_UK = [I | 0] returns q in the first d_nope columns and zeros after."""
    dn, dc, h = 8, 12, 3
    q = W.normal_bf16(21, 0x5555, 2 * 1 * h * dn).reshape(2, 1, h, dn)
    w = np.zeros((h, dn, dc), dtype=np.float32)
    for k in range(h):
        w[k, :, :dn] = np.eye(dn)
    out = orc.q_absorb(q, _bits(w))
    qv = W.bf16_bits_to_float32(q).astype(np.float64)
    assert np.array_equal(out[..., :dn], qv)
    assert not out[..., dn:].any()


def check_absorb_one_hot(orc):
    """q = e_d picks row d of that head's W_UK, exactly."""
    dn, dc, h = 16, 24, 2
    w = W.normal_bf16(22, 0x6666, h * dn * dc).reshape(h, dn, dc)
    q = np.zeros((1, 1, h, dn), dtype=np.float32)
    q[0, 0, 0, 5] = 1.0
    q[0, 0, 1, 11] = 1.0
    out = orc.q_absorb(_bits(q), w)
    wv = W.bf16_bits_to_float32(w).astype(np.float64)
    assert np.array_equal(out[0, 0, 0], wv[0, 5])
    assert np.array_equal(out[0, 0, 1], wv[1, 11])


def check_absorb_linear_and_head_relabel(orc):
    """Small-integer inputs keep every sum exact: absorb(q1 + q2) =
    absorb(q1) + absorb(q2), twice q gives twice the result, and relabelling
    the heads of q and W_UK together relabels the output."""
    rng = np.random.default_rng(23)
    dn, dc, h = 8, 10, 4
    q1 = rng.integers(-3, 4, (2, 2, h, dn)).astype(np.float32)
    q2 = rng.integers(-3, 4, (2, 2, h, dn)).astype(np.float32)
    w = rng.integers(-3, 4, (h, dn, dc)).astype(np.float32)
    a = orc.q_absorb(_bits(q1), _bits(w))
    b = orc.q_absorb(_bits(q2), _bits(w))
    ab = orc.q_absorb(_bits(q1 + q2), _bits(w))
    assert np.array_equal(ab, a + b)
    assert np.array_equal(orc.q_absorb(_bits(2 * q1), _bits(w)), 2 * a)
    perm = np.array([2, 0, 3, 1])
    pr = orc.q_absorb(_bits(q1[:, :, perm]), _bits(w[perm]))
    assert np.array_equal(pr, a[:, :, perm])
    assert not orc.q_absorb(_bits(np.zeros_like(q1)), _bits(w)).any()


ALL_CHECKS = [check_append_hand_slots, check_append_single_token,
              check_append_rejects_out_of_range, check_append_then_gather,
              check_absorb_hand_example, check_absorb_identity, check_absorb_one_hot,
              check_absorb_linear_and_head_relabel]
