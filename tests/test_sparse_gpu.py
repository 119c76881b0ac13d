"""Sparse decode (listed token positions) on the GPU against the fp64 oracle.

Same tolerances as the dense path (max |out err| <= 1e-2, max |lse err| <=
1e-3, empty rows exactly 0 / -inf, no NaN); rows that see only a few keys
are held to the bound the bf16 probabilities allow, as in the dense tests.
The identity list (position j at slot j, count = length) must reproduce the
dense kernel bit for bit: both then stage the same rows in the same layout.
"""
import numpy as np
import pytest

from mla_decode_attention_07_gb300 import libmla
from mla_decode_attention_07_gb300 import workloads as W
from test_parity_gpu import LSE_TOL, assert_parity, run_gpu, to_device, torch_cuda  # noqa: F401

pytestmark = pytest.mark.gpu


def run_sparse(torch, si, check_err=True):
    inp = si.base
    d = to_device(torch, inp)
    dev = torch.device("cuda", 0)
    idx = torch.from_numpy(np.ascontiguousarray(si.indices)).to(dev)
    cnt = torch.from_numpy(np.ascontiguousarray(si.counts)).to(dev)
    B, h_q = inp.batch, inp.h_q
    out = torch.full((B, 1, h_q, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((B, h_q, 1), float("nan"), dtype=torch.float32, device="cuda")
    meta, ws = libmla.alloc_plan_and_workspace(B, 1, h_q, 0)
    ws.fill_(float("nan"))
    libmla.mla_decode_plan(cnt, 1, h_q, meta)
    libmla.mla_decode_sparse(d["q"], d["kv"], d["bt"], d["sl"], idx, cnt, meta, out, lse,
                             inp.softmax_scale, ws)
    rc = libmla.mla_check_device_error()
    if check_err:
        assert rc == 0, libmla.mla_strerror(rc)
    return out.float().cpu().numpy(), lse.cpu().numpy(), rc


def sparse_rounding_bound(si, ref_o):
    """Elementwise bound on |out - exact| from bf16 P and bf16 out over the
    selected rows (see the dense tests' bf16_rounding_bound)."""
    inp = si.base
    v = (inp.kv_cache.view(np.uint16).astype(np.uint32) << 16).view(np.float32)[:, :, 0, :512]
    bound = np.zeros_like(ref_o)
    for b in range(inp.batch):
        c = int(si.counts[b])
        if c == 0:
            continue
        ts = si.indices[b, :c]
        rows = v[inp.block_table[b, ts // 64], ts % 64]
        vmax = np.abs(rows).max(axis=0).astype(np.float64)
        o = np.abs(ref_o[b])
        bound[b] = 2.0 ** -8 * (vmax + o) + 2.0 ** -9 * o + 1e-5
    return bound


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
    out, lse, _ = run_sparse(torch_cuda, si)
    ref_o, ref_l = oracle_mod.mla_decode_sparse(si)
    assert not np.isnan(out).any() and not np.isnan(lse).any()
    assert np.array_equal(np.isneginf(lse), np.isneginf(ref_l)), "-inf pattern differs"
    err = np.abs(out.astype(np.float64) - ref_o)
    bound = np.maximum(sparse_rounding_bound(si, ref_o), 1e-2)
    assert (err <= bound).all(), f"case {seed}: max err/bound {float((err / bound).max()):.3f}"
    fin = ~np.isneginf(ref_l)
    if fin.any():
        assert np.abs(lse[fin] - ref_l[fin]).max() <= LSE_TOL


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
