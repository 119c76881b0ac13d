"""Seeded input generators (CPU only)."""
import numpy as np
import pytest

from mla_decode_attention_07_gb300 import workloads as W


def test_splitmix64_published_vector():
    # First outputs of SplitMix64 seeded with 1234567 (the sequence printed with
    # the reference C implementation by Vigna) and with 0.
    assert [int(x) for x in W.splitmix64(1234567, 0, 5)] == [
        6457827717110365317, 3203168211198807973, 9817491932198370423,
        4593380528125082431, 16408922859458223821]
    assert int(W.splitmix64(0, 0, 1)[0]) == 0xE220A8397B1DCDAF


def test_splitmix64_counter_form_is_a_stream():
    a = W.splitmix64(77, 0, 100)
    b = np.concatenate([W.splitmix64(77, 0, 37), W.splitmix64(77, 37, 63)])
    assert np.array_equal(a, b)


def test_bf16_rounding_matches_torch():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(100000).astype(np.float32),
                        np.array([1.0, -2.5, 1.00390625, 1.01171875, 3.0e38, 1e-40],
                                 dtype=np.float32)])
    ours = W.float32_to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


def test_normals_moments_and_determinism():
    a = W.normal_bf16(5, W.TENSOR_KV, 1 << 18)
    b = W.normal_bf16(5, W.TENSOR_KV, 1 << 18, chunk=1000)
    assert np.array_equal(a, b)
    x = W.bf16_bits_to_float32(a).astype(np.float64)
    assert abs(x.mean()) < 0.01 and abs(x.std() - 1.0) < 0.01
    assert not np.array_equal(a, W.normal_bf16(6, W.TENSOR_KV, 1 << 18))


def test_permutation_is_a_permutation():
    p = W.permutation(3, W.TENSOR_PERM, 1000)
    assert sorted(p.tolist()) == list(range(1000))


def test_make_inputs_layout_and_poison():
    inp = W.make_inputs(9, 3, 2, 16, [65, 0, 128], extra_pages=2)
    assert inp.q.shape == (3, 2, 16, 576) and inp.kv_cache.shape == (6, 64, 1, 576)
    live = inp.block_table[0, :2].tolist() + inp.block_table[2, :2].tolist()
    assert len(set(live)) == 4
    assert np.all(inp.block_table[1] == inp.block_table[1, 0]) and inp.block_table[1, 0] not in live
    last = inp.block_table[0, 1]
    assert np.all(inp.kv_cache[last, 1:] == W.BF16_NAN)      # tail after token 64
    assert not np.any(inp.kv_cache[last, 0] == W.BF16_NAN)
    decoys = sorted(set(range(6)) - set(live))
    for p in decoys:
        assert np.all(inp.kv_cache[p] == W.BF16_NAN)


def test_workload_accounting():
    w = W.WORKLOADS["b16_h128_l4096"]
    assert abs(w.flops() / 1e9 - 18.25) < 0.01
    assert w.visible_keys() == 16 * 4096
    s = W.WORKLOADS["spec_b132_sq2_h128_l8192"]
    assert s.visible_keys() == 132 * (8192 + 8191)
    r = W.WORKLOADS["ragged_b64_h128"].seqlens()
    assert r.min() >= 1 and r.max() <= 8192 and len(r) == 64


def test_sparse_positions_are_a_seeded_subset():
    idx, cnt = W.draw_indices(9, [300, 64, 5, 0], 128)
    assert list(cnt) == [128, 64, 5, 0]
    for b, (L, c) in enumerate([(300, 128), (64, 64), (5, 5), (0, 0)]):
        sel = idx[b, :c]
        assert len(set(sel.tolist())) == c                  # distinct
        assert ((sel >= 0) & (sel < max(L, 1))).all()
        assert (idx[b, c:] == -1).all()
    assert sorted(idx[1, :64].tolist()) == list(range(64))  # count == L: a permutation
    again, _ = W.draw_indices(9, [300, 64, 5, 0], 128)
    assert np.array_equal(idx, again)                       # seeded
    other, _ = W.draw_indices(10, [300, 64, 5, 0], 128)
    assert not np.array_equal(idx, other)


def test_sparse_repeats_and_bad_counts():
    idx, cnt = W.draw_indices(3, [10], 40, counts=[40], repeats=True)
    assert cnt[0] == 40 and ((idx[0] >= 0) & (idx[0] < 10)).all()
    with pytest.raises(ValueError):
        W.draw_indices(3, [10], 40, counts=[20])            # 20 distinct of 10
    with pytest.raises(ValueError):
        W.draw_indices(3, [100], 8, counts=[9])             # more than top-k


def test_sparse_pool_block_tables_stay_in_the_pool():
    si = W.make_sparse_inputs(4, 3, 16, [1000, 65, 64], 32, pool_pages=7)
    assert si.base.kv_cache.shape == (7, W.PAGE, 1, W.D_QK)
    assert si.base.block_table.shape == (3, 16)
    assert ((si.base.block_table >= 0) & (si.base.block_table < 7)).all()
    assert si.base.q.shape == (3, 1, 16, W.D_QK)


def test_step_generators_shapes_and_determinism():
    p1 = W.make_prologue_inputs(3, 2, 2, 16, [100, 70])
    p2 = W.make_prologue_inputs(3, 2, 2, 16, [100, 70])
    assert p1.kv_new.shape == (2, 2, W.D_QK) and p1.q_nope.shape == (2, 2, 16, W.D_NOPE)
    assert p1.q_rope.shape == (2, 2, 16, W.D_ROPE) and p1.w_uk.shape == (16, W.D_NOPE, W.D_C)
    assert np.array_equal(p1.w_uk, p2.w_uk) and np.array_equal(p1.kv_new, p2.kv_new)
    std = float(W.bf16_bits_to_float32(p1.w_uk).std())
    assert abs(std - W.D_NOPE ** -0.5) < 0.01


def test_normal_f16_is_rounded_from_the_float32_stream():
    a = W.normal_f16(6, W.TENSOR_GEMM_A, 4096)
    v = a.view(np.float16).astype(np.float64)
    assert abs(v.mean()) < 0.1 and abs(v.std() - 1.0) < 0.05
    # rounding float16 -> float32 -> float16 is the identity on these bits
    assert np.array_equal(v.astype(np.float32).astype(np.float16).view(np.uint16), a)
    assert np.array_equal(W.normal_f16(6, W.TENSOR_GEMM_A, 10), a[:10])
