"""Dense attention forward on the GPU against the fp64 oracle (needs a
GB300).

Bar: the decode path's fixed tolerances, max |out - oracle| <= 1e-2 over
every element (bf16 output upcast) and max |lse - oracle| <= 1e-3; nothing
may be NaN.  Each case first checks on the CPU that its exact result can be
written in bf16 within 1e-2 at all (values of magnitude 4 and more can sit
up to 2^-6 from the nearest bf16), so that the bar is attainable.
"""
import numpy as np
import pytest

from mla_decode_attention_07_gb300 import libmla
from mla_decode_attention_07_gb300 import workloads as W

pytestmark = pytest.mark.gpu

OUT_TOL = 1e-2
LSE_TOL = 1e-3


@pytest.fixture(scope="module")
def torch_cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    return torch


def run_attention(torch, ai):
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a.view(np.int16))).to("cuda").view(
        torch.bfloat16)
    B, S, H, _ = ai.q.shape
    dv = ai.v.shape[3]
    out = torch.full((B, S, H, dv), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((B, H, S), float("nan"), dtype=torch.float32, device="cuda")
    libmla.mla_attention_fwd(t(ai.q), t(ai.k), t(ai.v), out, lse, ai.causal, ai.scale)
    rc = libmla.mla_check_device_error()
    assert rc == 0, libmla.mla_strerror(rc)
    return out.float().cpu().numpy(), lse.cpu().numpy()


def bf16_round_error(x):
    r = W.bf16_bits_to_float32(W.float32_to_bf16_bits(np.asarray(x, dtype=np.float32)))
    return float(np.abs(r.astype(np.float64) - x).max())


CASES = [
    # seed, batch, seqlen, heads, d_qk, causal
    (401, 1, 128, 1, 128, True),
    (402, 2, 200, 3, 64, True),        # a ragged second query tile
    (403, 1, 300, 2, 192, False),
    (404, 2, 1000, 4, 192, True),      # eight query tiles, the causal diagonal in each
    (405, 1, 129, 8, 128, False),
    (406, 1, 1, 2, 64, True),          # one token
    (407, 3, 513, 2, 192, True),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"s{c[0]}_b{c[1]}_s{c[2]}_h{c[3]}_d{c[4]}"
                         f"_{'causal' if c[5] else 'full'}")
def test_attention_parity(torch_cuda, case, oracle_mod):
    seed, B, S, H, dqk, causal = case
    ai = W.make_attention_inputs(seed, B, S, H, dqk, 128, causal)
    ref_o, ref_l = oracle_mod.attention(ai)
    assert bf16_round_error(ref_o) <= OUT_TOL, "bar not attainable in bf16 for this case"
    out, lse = run_attention(torch_cuda, ai)
    assert not np.isnan(out).any() and not np.isnan(lse).any()
    eo = float(np.abs(out - ref_o).max())
    el = float(np.abs(lse - ref_l).max())
    assert eo <= OUT_TOL, f"max|out err| {eo:.3e}"
    assert el <= LSE_TOL, f"max|lse err| {el:.3e}"


def test_attention_output_only_16_byte_aligned(torch_cuda, oracle_mod):
    """out placed 16 bytes into a larger buffer (16- but not 32-byte
    aligned), which takes the kernel's 16-byte store path; the words around
    it stay untouched."""
    ai = W.make_attention_inputs(408, 2, 300, 3, 192, 128, True)
    ref_o, ref_l = oracle_mod.attention(ai)
    t = lambda a: torch_cuda.from_numpy(np.ascontiguousarray(a.view(np.int16))).to("cuda").view(
        torch_cuda.bfloat16)
    n = 2 * 300 * 3 * 128
    buf = torch_cuda.full((n + 32,), 7.0, dtype=torch_cuda.bfloat16, device="cuda")
    out = buf[8:8 + n].view(2, 300, 3, 128)
    assert out.data_ptr() % 32 == 16
    lse = torch_cuda.empty((2, 3, 300), dtype=torch_cuda.float32, device="cuda")
    libmla.mla_attention_fwd(t(ai.q), t(ai.k), t(ai.v), out, lse, ai.causal, ai.scale)
    assert libmla.mla_check_device_error() == 0
    b = buf.float().cpu().numpy()
    assert (b[:8] == 7.0).all() and (b[8 + n:] == 7.0).all()
    assert float(np.abs(out.float().cpu().numpy() - ref_o).max()) <= OUT_TOL
    assert float(np.abs(lse.cpu().numpy() - ref_l).max()) <= LSE_TOL


def test_attention_prefill_workload_sampled(torch_cuda, oracle_mod):
    """The MLA-prefill workload at full size through the call the benchmark
    times, 256 sampled rows (and the corners) against the oracle."""
    w = W.ATTENTION_WORKLOADS["prefill_b1_h128_s4096_d192"]
    ai = w.make()
    out, lse = run_attention(torch_cuda, ai)
    rng = np.random.default_rng(9)
    rows = np.stack([rng.integers(0, w.batch, 256), rng.integers(0, w.heads, 256),
                     rng.integers(0, w.seqlen, 256)], axis=1)
    rows = np.concatenate([[[0, 0, 0], [0, w.heads - 1, w.seqlen - 1]], rows]).astype(np.int32)
    ref_o, ref_l = oracle_mod.attention_rows(ai, rows)
    got_o = out[rows[:, 0], rows[:, 2], rows[:, 1]]
    got_l = lse[rows[:, 0], rows[:, 1], rows[:, 2]]
    assert float(np.abs(got_o - ref_o).max()) <= OUT_TOL
    assert float(np.abs(got_l - ref_l).max()) <= LSE_TOL
    assert not np.isnan(out).any() and not np.isnan(lse).any()


MULTI_ITEM_CASES = [
    # seed, batch, seqlen, heads, d_qk, causal: several work items per CTA
    # (query tiles x heads x batch well above the SM count), so each CTA runs
    # item switches (the next item's Q staged during the previous one)
    (409, 3, 1500, 40, 192, True),     # 1440 items, ragged last query tile
    (410, 2, 1100, 72, 128, False),    # 1296 items, full rows
]


@pytest.mark.parametrize("case", MULTI_ITEM_CASES,
                         ids=lambda c: f"s{c[0]}_b{c[1]}_s{c[2]}_h{c[3]}_d{c[4]}"
                         f"_{'causal' if c[5] else 'full'}")
def test_attention_many_items_per_cta_sampled(torch_cuda, case, oracle_mod):
    seed, B, S, H, dqk, causal = case
    ai = W.make_attention_inputs(seed, B, S, H, dqk, 128, causal)
    out, lse = run_attention(torch_cuda, ai)
    rng = np.random.default_rng(seed)
    rows = np.stack([rng.integers(0, B, 192), rng.integers(0, H, 192), rng.integers(0, S, 192)],
                    axis=1)
    corners = [[0, 0, 0], [B - 1, H - 1, S - 1], [B - 1, 0, S - 1], [0, H - 1, 127], [0, 1, 128]]
    rows = np.concatenate([corners, rows]).astype(np.int32)
    ref_o, ref_l = oracle_mod.attention_rows(ai, rows)
    got_o = out[rows[:, 0], rows[:, 2], rows[:, 1]]
    got_l = lse[rows[:, 0], rows[:, 1], rows[:, 2]]
    assert not np.isnan(out).any() and not np.isnan(lse).any()
    assert float(np.abs(got_o - ref_o).max()) <= OUT_TOL
    assert float(np.abs(got_l - ref_l).max()) <= LSE_TOL
