"""Pins of the GEMM oracle (gemm_oracle.c).

Each check takes an ``oracle.Gemm`` and raises AssertionError when the oracle
disagrees with something fixed independently of its code: the IEEE binary16
values of chosen bit patterns, an identity or one-hot factor, all-ones
factors (C = K), and a small product worked by hand.
"""
import numpy as np

F16, BF16 = 0, 1


def _f16(x):
    return np.asarray(x, dtype=np.float16).view(np.uint16)


def check_f16_values(orc):
    """1 x 1 x 1 products with B = 1 return A's value: 1, -2, the largest
    finite value 65504, the smallest normal 2^-14, the smallest subnormal
    2^-24, a subnormal 3 * 2^-24, and 1 + 2^-10."""
    one = np.array([[0x3C00]], dtype=np.uint16)
    for bits, val in ((0x3C00, 1.0), (0xC000, -2.0), (0x7BFF, 65504.0), (0x0400, 2.0 ** -14),
                      (0x0001, 2.0 ** -24), (0x0003, 3 * 2.0 ** -24), (0x3C01, 1 + 2.0 ** -10)):
        c = orc.gemm(np.array([[bits]], dtype=np.uint16), one, F16)
        assert c[0, 0] == val, (hex(bits), c[0, 0], val)


def check_bf16_values(orc):
    one = np.array([[0x3F80]], dtype=np.uint16)
    for bits, val in ((0x3F80, 1.0), (0xC040, -3.0), (0x3F81, 1 + 2.0 ** -7)):
        c = orc.gemm(np.array([[bits]], dtype=np.uint16), one, BF16)
        assert c[0, 0] == val


def check_hand_product(orc):
    """[[1, 2, 3], [4, 5, 6]] x [[1, -1], [0, 2], [0.5, 1]] = [[2.5, 6], [7, 12]]."""
    a = _f16([[1, 2, 3], [4, 5, 6]])
    b = _f16([[1, -1], [0, 2], [0.5, 1]])
    assert np.array_equal(orc.gemm(a, b, F16), np.array([[2.5, 6.0], [7.0, 12.0]]))


def check_identity_and_one_hot(orc):
    rng = np.random.default_rng(31)
    n = 24
    b = _f16(rng.standard_normal((n, n)))
    bv = b.view(np.float16).astype(np.float64)
    assert np.array_equal(orc.gemm(_f16(np.eye(n)), b, F16), bv)
    a = np.zeros((5, n), dtype=np.float32)
    a[3, 7] = 1.0
    c = orc.gemm(_f16(a), b, F16)
    assert np.array_equal(c[3], bv[7]) and not np.delete(c, 3, axis=0).any()


def check_ones(orc):
    """All-ones factors of a non-square shape: every entry is K."""
    M, K, N = 7, 33, 5
    c = orc.gemm(_f16(np.ones((M, K))), _f16(np.ones((K, N))), F16)
    assert c.shape == (M, N) and np.all(c == K)


def check_entries_match_whole(orc):
    rng = np.random.default_rng(32)
    M, K, N = 9, 17, 11
    a = _f16(rng.integers(-4, 5, (M, K)))
    b = _f16(rng.integers(-4, 5, (K, N)))
    whole = orc.gemm(a, b, F16)
    ent = np.array([[0, 0], [8, 10], [3, 4], [8, 0]], dtype=np.int32)
    assert np.array_equal(orc.gemm_entries(a, b, F16, ent), whole[ent[:, 0], ent[:, 1]])
    # integers: every product and sum is exact, so this is the exact product
    assert np.array_equal(whole, a.view(np.float16).astype(np.int64) @
                          b.view(np.float16).astype(np.int64))


ALL_CHECKS = [check_f16_values, check_bf16_values, check_hand_product,
              check_identity_and_one_hot, check_ones, check_entries_match_whole]
