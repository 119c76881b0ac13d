"""The steps before the decode call and the tensor-core GEMM on the GPU,
against the CPU oracles (needs a GB300).

Bars:
* cache append: bit for bit, the whole cache compared.
* query absorption: the latent part is a 128-term fp32 sum rounded to bf16,
  so |gpu - exact| <= half a bf16 unit in the last place (2^(e - 8) for
  |value| in [2^e, 2^(e+1))) + 2^-16 S, S = sum_d |q_d w_dc| (twice the
  worst-case fp32 accumulation error of 128 terms, 128 * 2^-24 = 2^-17),
  element by element; the rotary part is a bit-exact copy.
* GEMM: the GEMM tutorial's bar, relative error ||C - exact||_F /
  ||exact||_F < 2e-2, and element by element the bound the arithmetic gives:
  half a unit in the last place of the output type at |exact| plus 2 K
  2^-24 S, S = sum_k |a_k b_k|.
"""
import numpy as np
import pytest

from mla_decode_attention_07_gb300 import libmla
from mla_decode_attention_07_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch_cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    return torch


def _dev(torch, a, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a)).to("cuda")
    return t.view(dtype) if dtype is not None else t


APPEND_CASES = [
    # seed, batch, s_q, seqlens, extra_pages
    (301, 1, 1, [1], 0),
    (302, 3, 1, [64, 65, 4096], 2),
    (303, 4, 2, [2, 63, 64, 130], 1),
    (304, 16, 1, [4096] * 16, 0),
    (305, 132, 2, list(W.uniform_int(305, W.TENSOR_SEQLENS, 132, 2, 8192)), 3),
]


@pytest.mark.parametrize("case", APPEND_CASES, ids=lambda c: f"s{c[0]}_b{c[1]}_sq{c[2]}")
def test_cache_append_bit_exact(torch_cuda, case, oracle_mod):
    seed, B, s_q, seqlens, extra = case
    p = W.make_prologue_inputs(seed, B, s_q, 16, seqlens, extra_pages=extra)
    base = p.base
    want = oracle_mod.cache_append(p.kv_new, base.kv_cache, base.block_table,
                                   base.cache_seqlens)
    kv = _dev(torch_cuda, base.kv_cache.view(np.int16), torch_cuda.bfloat16)
    libmla.mla_cache_append(_dev(torch_cuda, p.kv_new.view(np.int16), torch_cuda.bfloat16), kv,
                            _dev(torch_cuda, base.block_table),
                            _dev(torch_cuda, base.cache_seqlens))
    assert libmla.mla_check_device_error() == 0
    got = kv.view(torch_cuda.int16).cpu().numpy().view(np.uint16)
    assert np.array_equal(got, want)


def test_cache_append_out_of_range_is_flagged(torch_cuda):
    p = W.make_prologue_inputs(306, 2, 2, 16, [1, 100])        # entry 0: 1 token, 2 new
    base = p.base
    kv = _dev(torch_cuda, base.kv_cache.view(np.int16), torch_cuda.bfloat16)
    libmla.mla_check_device_error()
    libmla.mla_cache_append(_dev(torch_cuda, p.kv_new.view(np.int16), torch_cuda.bfloat16), kv,
                            _dev(torch_cuda, base.block_table),
                            _dev(torch_cuda, base.cache_seqlens))
    assert libmla.mla_check_device_error() == libmla.MLA_ERR_DEVICE_BOUNDS


def _abs_bits16(bits):
    return (np.asarray(bits, dtype=np.uint16) & np.uint16(0x7FFF)).astype(np.uint16)


ABSORB_CASES = [
    # seed, batch, s_q, h_q
    (311, 1, 1, 16),
    (312, 3, 2, 128),
    (313, 16, 1, 128),           # the batch-16 decode shape
    (314, 200, 1, 32),           # two row tiles, the second ragged
    (315, 132, 2, 128),          # the speculative decode shape: three row tiles
    (317, 129, 1, 3),            # two row tiles of 80, the second ragged
    (318, 1, 1, 1),              # one row, one head
    (319, 300, 3, 4),            # 900 rows: eight tiles of 128, the last holding 4 rows
]


@pytest.mark.parametrize("case", ABSORB_CASES, ids=lambda c: f"s{c[0]}_b{c[1]}_sq{c[2]}_h{c[3]}")
def test_q_absorb_parity(torch_cuda, case, oracle_mod):
    seed, B, s_q, h_q = case
    p = W.make_prologue_inputs(seed, B, s_q, h_q, [max(s_q, 64)] * B)
    bf = torch_cuda.bfloat16
    q = torch_cuda.full((B, s_q, h_q, W.D_QK), float("nan"), dtype=bf, device="cuda")
    libmla.mla_q_absorb(_dev(torch_cuda, p.q_nope.view(np.int16), bf),
                        _dev(torch_cuda, p.q_rope.view(np.int16), bf),
                        _dev(torch_cuda, p.w_uk.view(np.int16), bf), q)
    assert libmla.mla_check_device_error() == 0
    got = q.view(torch_cuda.int16).cpu().numpy().view(np.uint16)
    assert np.array_equal(got[..., W.D_C:], p.q_rope), "rotary part not copied bit for bit"
    exact = oracle_mod.q_absorb(p.q_nope, p.w_uk)
    mag = oracle_mod.q_absorb(_abs_bits16(p.q_nope), _abs_bits16(p.w_uk))
    lat = W.bf16_bits_to_float32(got[..., :W.D_C]).astype(np.float64)
    assert np.isfinite(lat).all()
    err = np.abs(lat - exact)
    acc = 2.0 ** -16 * mag
    bound = _ulp_half(np.abs(exact) + acc, "bf16") + acc + 1e-30
    assert (err <= bound).all(), f"max err/bound {float((err / bound).max()):.3f}"


def test_absorbed_query_decodes_like_the_oracle(torch_cuda, oracle_mod):
    """Append + absorption + decode chained on the GPU, against the oracle's
    decode of the oracle's appended cache and the GPU's (checked) query."""
    p = W.make_prologue_inputs(316, 4, 1, 128, [300, 64, 1000, 65], extra_pages=1)
    base = p.base
    bf = torch_cuda.bfloat16
    kv = _dev(torch_cuda, base.kv_cache.view(np.int16), bf)
    bt, sl = _dev(torch_cuda, base.block_table), _dev(torch_cuda, base.cache_seqlens)
    libmla.mla_cache_append(_dev(torch_cuda, p.kv_new.view(np.int16), bf), kv, bt, sl)
    q = torch_cuda.empty((4, 1, 128, W.D_QK), dtype=bf, device="cuda")
    libmla.mla_q_absorb(_dev(torch_cuda, p.q_nope.view(np.int16), bf),
                        _dev(torch_cuda, p.q_rope.view(np.int16), bf),
                        _dev(torch_cuda, p.w_uk.view(np.int16), bf), q)
    out = torch_cuda.empty((4, 1, 128, 512), dtype=torch_cuda.float32, device="cuda")
    lse = torch_cuda.empty((4, 128, 1), dtype=torch_cuda.float32, device="cuda")
    meta, ws = libmla.alloc_plan_and_workspace(4, 1, 128, 0)
    libmla.mla_decode_plan(sl, 1, 128, meta)
    libmla.mla_decode_f32(q, kv, bt, sl, meta, out, lse, W.SOFTMAX_SCALE, ws)
    assert libmla.mla_check_device_error() == 0
    cache = oracle_mod.cache_append(p.kv_new, base.kv_cache, base.block_table,
                                    base.cache_seqlens)
    qb = q.view(torch_cuda.int16).cpu().numpy().view(np.uint16)
    inp = W.DecodeInputs(q=qb, kv_cache=cache, block_table=base.block_table,
                         cache_seqlens=base.cache_seqlens, s_q=1, h_q=128)
    ref_o, ref_l = oracle_mod.mla_decode(inp)
    assert float(np.abs(out.cpu().numpy() - ref_o).max()) <= 1e-2
    assert float(np.abs(lse.cpu().numpy() - ref_l).max()) <= 1e-3


def _f16(torch, bits):
    return _dev(torch, bits.view(np.int16), torch.float16)


def _ulp_half(exact, out):
    """Half a unit in the last place of the output type at |exact|."""
    a = np.maximum(np.abs(exact), 1e-30)
    e = np.floor(np.log2(a))
    if out == "f16":
        return np.ldexp(1.0, (np.maximum(e, -14) - 11).astype(np.int64))
    if out == "bf16":
        return np.ldexp(1.0, (e - 8).astype(np.int64))
    return np.ldexp(1.0, (e - 24).astype(np.int64))


def _check_gemm(exact, mag, got, K, out):
    assert np.isfinite(got).all()
    rel = float(np.linalg.norm(got - exact) / max(np.linalg.norm(exact), 1e-30))
    assert rel < 2e-2, f"relative error {rel:.3e}"
    err = np.abs(got - exact)
    acc = 2.0 * K * 2.0 ** -24 * mag
    bound = _ulp_half(np.abs(exact) + acc, out) + acc + 1e-30
    assert (err <= bound).all(), f"max err/bound {float((err / bound).max()):.3f}"
    return rel


GEMM_CASES = [
    # seed, M, N, K, in, out
    (321, 256, 256, 256, "f16", "f16"),
    (322, 300, 200, 136, "f16", "f32"),       # ragged in M, N and K
    (323, 128, 512, 1024, "bf16", "bf16"),
    (324, 1, 8, 8, "f16", "f16"),
    (325, 1000, 768, 520, "f16", "f16"),
]


@pytest.mark.parametrize("case", GEMM_CASES, ids=lambda c: f"s{c[0]}_{c[1]}x{c[2]}x{c[3]}_{c[4]}_{c[5]}")
def test_gemm_parity(torch_cuda, case, oracle_mod):
    seed, M, N, K, tin, tout = case
    if tin == "f16":
        a = W.normal_f16(seed, W.TENSOR_GEMM_A, M * K).reshape(M, K)
        b = W.normal_f16(seed, W.TENSOR_GEMM_B, K * N).reshape(K, N)
        da, db = _f16(torch_cuda, a), _f16(torch_cuda, b)
    else:
        a = W.normal_bf16(seed, W.TENSOR_GEMM_A, M * K).reshape(M, K)
        b = W.normal_bf16(seed, W.TENSOR_GEMM_B, K * N).reshape(K, N)
        da = _dev(torch_cuda, a.view(np.int16), torch_cuda.bfloat16)
        db = _dev(torch_cuda, b.view(np.int16), torch_cuda.bfloat16)
    tdt = {"f16": torch_cuda.float16, "bf16": torch_cuda.bfloat16, "f32": torch_cuda.float32}[tout]
    c = torch_cuda.full((M, N), float("nan"), dtype=tdt, device="cuda")
    libmla.mla_gemm(da, db, c)
    assert libmla.mla_check_device_error() == 0
    fmt = 0 if tin == "f16" else 1
    exact = oracle_mod.gemm(a, b, fmt)
    mag = oracle_mod.gemm(_abs_bits16(a), _abs_bits16(b), fmt)
    _check_gemm(exact, mag, c.float().cpu().numpy().astype(np.float64), K, tout)


def test_gemm_2048_sampled(torch_cuda, oracle_mod):
    """The tutorial's FP16 2048^3 GEMM through the call the benchmark times:
    8192 sampled entries (and the corners) against the oracle."""
    w = W.GEMM_WORKLOADS["gemm_f16_2048"]
    a, b = w.make()
    c = torch_cuda.empty((w.M, w.N), dtype=torch_cuda.float16, device="cuda")
    libmla.mla_gemm(_f16(torch_cuda, a), _f16(torch_cuda, b), c)
    assert libmla.mla_check_device_error() == 0
    got = c.float().cpu().numpy().astype(np.float64)
    rng = np.random.default_rng(7)
    ent = np.stack([rng.integers(0, w.M, 8192), rng.integers(0, w.N, 8192)], axis=1)
    ent = np.concatenate([[[0, 0], [w.M - 1, w.N - 1], [0, w.N - 1], [w.M - 1, 0]], ent])
    ent = ent.astype(np.int32)
    exact = oracle_mod.gemm_entries(a, b, 0, ent)
    mag = oracle_mod.gemm_entries(_abs_bits16(a), _abs_bits16(b), 0, ent)
    _check_gemm(exact, mag, got[ent[:, 0], ent[:, 1]], w.K, "f16")
    assert np.isfinite(got).all()
