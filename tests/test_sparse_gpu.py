"""Sparse decode (listed token positions) on the GPU against the fp64 oracle.

Same fixed tolerances as the dense path (max |out err| <= 1e-2, max |lse err|
<= 1e-3, empty rows exactly 0 / -inf, no NaN), for the fp32 output and for
the bf16 output, which must be the fp32 output rounded to nearest even.
The identity list (position j at slot j, count = length) must reproduce the
dense kernel bit for bit: both then stage the same rows in the same layout.
"""
import numpy as np
import pytest

from mla_decode_attention_07_gb300 import libmla
from mla_decode_attention_07_gb300 import workloads as W
from test_parity_gpu import (assert_bf16_is_rounded_f32, assert_parity, run_gpu,  # noqa: F401
                             to_device, torch_cuda)

pytestmark = pytest.mark.gpu


def run_sparse(torch, si, check_err=True, out_f32=False):
    inp = si.base
    d = to_device(torch, inp)
    dev = torch.device("cuda", 0)
    idx = torch.from_numpy(np.ascontiguousarray(si.indices)).to(dev)
    cnt = torch.from_numpy(np.ascontiguousarray(si.counts)).to(dev)
    B, h_q = inp.batch, inp.h_q
    odt = torch.float32 if out_f32 else torch.bfloat16
    out = torch.full((B, 1, h_q, 512), float("nan"), dtype=odt, device="cuda")
    lse = torch.full((B, h_q, 1), float("nan"), dtype=torch.float32, device="cuda")
    meta, ws = libmla.alloc_plan_and_workspace(B, 1, h_q, 0)
    ws.fill_(float("nan"))
    libmla.mla_decode_plan(cnt, 1, h_q, meta)
    fn = libmla.mla_decode_sparse_f32 if out_f32 else libmla.mla_decode_sparse
    fn(d["q"], d["kv"], d["bt"], d["sl"], idx, cnt, meta, out, lse, inp.softmax_scale, ws)
    rc = libmla.mla_check_device_error()
    if check_err:
        assert rc == 0, libmla.mla_strerror(rc)
    return out.float().cpu().numpy(), lse.cpu().numpy(), rc


SPARSE_SMALL = [
    # seed, h_q, seqlens, topk, counts, repeats
    (201, 128, [300, 64, 1], 128, None, False),
    (202, 16, [1000, 200], 100, [100, 37], False),       # topk not a multiple of 64
    (203, 64, [90, 40, 500], 64, [64, 0, 64], True),     # repeated positions, an empty entry
    (204, 128, [20000, 20000], 2048, None, False),       # 32 chunks: split over clusters
    (205, 128, [5000] * 16, 512, None, False),
    (207, 32, list(W.uniform_int(207, W.TENSOR_SEQLENS, 40, 1, 3000)), 256, None, False),
]


@pytest.mark.parametrize("case", SPARSE_SMALL, ids=lambda c: f"s{c[0]}_h{c[1]}_k{c[3]}")
def test_sparse_small_parity(torch_cuda, case, oracle_mod):
    seed, h_q, seqlens, topk, counts, repeats = case
    si = W.make_sparse_inputs(seed, len(seqlens), h_q, seqlens, topk, counts, repeats=repeats)
    ref_o, ref_l = oracle_mod.mla_decode_sparse(si)
    out32, lse32, _ = run_sparse(torch_cuda, si, out_f32=True)
    assert_parity(out32, lse32, ref_o, ref_l, f"sparse case {seed} fp32 out")
    out16, lse16, _ = run_sparse(torch_cuda, si)
    assert np.array_equal(lse16, lse32)
    assert_bf16_is_rounded_f32(out16, out32, f"sparse case {seed}")
    assert_parity(out16, lse16, ref_o, ref_l, f"sparse case {seed} bf16 out")


def test_sparse_identity_list_is_dense(torch_cuda):
    inp = W.make_inputs(206, 3, 1, 128, [300, 64, 129], extra_pages=1)
    topk = 320
    idx = np.full((3, topk), -1, dtype=np.int32)
    for b in range(3):
        L = int(inp.cache_seqlens[b])
        idx[b, :L] = np.arange(L)
    si = W.SparseInputs(base=inp, indices=idx, counts=inp.cache_seqlens.copy())
    so, sl_, _ = run_sparse(torch_cuda, si)
    do, dl, _ = run_gpu(torch_cuda, inp)
    assert np.array_equal(so, do) and np.array_equal(sl_, dl)


def test_sparse_bad_position_is_flagged(torch_cuda):
    si = W.make_sparse_inputs(208, 2, 16, [100, 100], 64)
    si.indices[1, 5] = 100                     # == cache length: past the sequence
    _, _, rc = run_sparse(torch_cuda, si, check_err=False)
    assert rc == libmla.MLA_ERR_DEVICE_BOUNDS


def test_sparse_workload_sampled(torch_cuda, oracle_mod):
    """The 128K-context workload at full size, 64 sampled rows."""
    w = W.SPARSE_WORKLOADS["sparse_b64_h128_l131072_k2048"]
    si = w.make()
    out, lse, _ = run_sparse(torch_cuda, si)
    rng = np.random.default_rng(5)
    rows = np.stack([rng.integers(0, w.batch, 62), rng.integers(0, w.h_q, 62)], axis=1)
    rows = np.concatenate([[[0, 0], [w.batch - 1, w.h_q - 1]], rows]).astype(np.int32)
    ref_o, ref_l = oracle_mod.mla_decode_sparse_rows(si, rows)
    got_o = out[rows[:, 0], 0, rows[:, 1]]
    got_l = lse[rows[:, 0], rows[:, 1], 0]
    assert_parity(got_o, got_l, ref_o, ref_l, "sparse workload")
    assert not np.isnan(out).any() and not np.isnan(lse).any()
