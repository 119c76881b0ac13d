"""CUDA path against the fp64 oracle, element by element (needs a GB300).

Tolerance, fixed: max |out - oracle| <= 1e-2 over every output element and
max |lse - oracle| <= 1e-3; rows with no visible key must give out = 0 and
lse = -inf exactly, and nothing may be NaN.  Every small case runs twice:
with the fp32 output (mla_decode_f32), which is held to the bar, and with the
bf16 output (mla_decode), which must be exactly the fp32 output rounded to
nearest even and is held to the bar as well, except on the one case whose
exact result cannot be written in bf16 within 1e-2 at all (case 112: the
fp64 oracle's own output rounded to bf16 misses it, as
tests/test_output_format.py shows on the CPU).
"""
import numpy as np
import pytest

import plan_model
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


def to_device(torch, inp):
    dev = torch.device("cuda", 0)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)
    return dict(q=t(inp.q.view(np.int16)).view(torch.bfloat16),
                kv=t(inp.kv_cache.view(np.int16)).view(torch.bfloat16),
                bt=t(inp.block_table), sl=t(inp.cache_seqlens))


def run_gpu(torch, inp, d=None, check_err=True, out_f32=False):
    d = d or to_device(torch, inp)
    B, s_q, h_q = inp.batch, inp.s_q, inp.h_q
    odt = torch.float32 if out_f32 else torch.bfloat16
    out = torch.full((B, s_q, h_q, 512), float("nan"), dtype=odt, device="cuda")
    lse = torch.full((B, h_q, s_q), float("nan"), dtype=torch.float32, device="cuda")
    meta, ws = libmla.alloc_plan_and_workspace(B, s_q, h_q, 0)
    ws.fill_(float("nan"))
    libmla.mla_decode_plan(d["sl"], s_q, h_q, meta)
    fn = libmla.mla_decode_f32 if out_f32 else libmla.mla_decode
    fn(d["q"], d["kv"], d["bt"], d["sl"], meta, out, lse, inp.softmax_scale, ws)
    rc = libmla.mla_check_device_error()
    if check_err:
        assert rc == 0, libmla.mla_strerror(rc)
    if out_f32:
        return out.cpu().numpy(), lse.cpu().numpy(), meta
    return out.float().cpu().numpy(), lse.cpu().numpy(), meta


def assert_bf16_is_rounded_f32(out_bf16, out_f32, what=""):
    """The bf16 output is the fp32 output rounded to nearest even, bit for bit."""
    want = W.float32_to_bf16_bits(np.ascontiguousarray(out_f32, dtype=np.float32))
    got = W.float32_to_bf16_bits(np.ascontiguousarray(out_bf16, dtype=np.float32))
    bad = int((want != got).sum())
    assert bad == 0, f"{what}: {bad} bf16 outputs are not the rounded fp32 outputs"


def assert_parity(out, lse, ref_o, ref_l, what=""):
    assert not np.isnan(out).any(), f"{what}: NaN in out"
    assert not np.isnan(lse).any(), f"{what}: NaN in lse"
    empty = np.isneginf(ref_l)
    assert np.array_equal(np.isneginf(lse), empty), f"{what}: -inf pattern differs"
    eo = float(np.abs(out - ref_o).max()) if out.size else 0.0
    el = float(np.abs(np.where(empty, 0.0, lse - ref_l)).max()) if lse.size else 0.0
    assert eo <= OUT_TOL, f"{what}: max|out err| {eo:.3e}"
    assert el <= LSE_TOL, f"{what}: max|lse err| {el:.3e}"
    return eo, el


SMALL = [
    # seed, batch, s_q, h_q, seqlens, extra_pages
    (101, 1, 1, 16, [256], 0),
    (102, 2, 1, 128, [64, 65], 1),
    (103, 3, 2, 128, [1, 127, 300], 2),
    (104, 4, 1, 64, [1000, 1, 63, 64], 1),
    (105, 2, 2, 16, [513, 2], 0),
    (106, 5, 1, 32, [0, 5, 129, 0, 700], 1),
    (107, 1, 1, 128, [3000], 0),
    (108, 2, 2, 64, [1, 1], 0),
    (109, 1, 1, 8, [77], 0),
    (110, 3, 2, 100, [333, 90, 1], 1),
    (111, 16, 1, 128, [640] * 16, 0),
    # many one-page entries: every cluster gets several tiles whose pages
    # alternate between the two page-worker sets (a tile can have no page of
    # one set), which exercises the running-max and sums hand-offs
    (112, 300, 1, 128, list(W.uniform_int(112, W.TENSOR_SEQLENS, 300, 1, 64)), 0),
    (113, 200, 2, 64, list(W.uniform_int(113, W.TENSOR_SEQLENS, 200, 0, 256)), 1),
    # more query tokens per entry: 4 x 64 rows (two tiles), 8 x 128 rows
    # (eight tiles, so eight groups of clusters), and a single head
    (114, 3, 4, 64, [300, 4, 1100], 1),
    (115, 2, 8, 128, [900, 2000], 0),
    (116, 3, 1, 1, [70, 1, 500], 1),
    # At most 16 query rows per entry with more than 4 block-table pages per
    # cluster run the narrow kernel (the CTA pair takes alternate pages and
    # merges per entry; cases 101, 109 and 116 above stay on the general
    # kernel).  Many short entries (several entries per cluster, one-page
    # segments where one CTA has no page, split and whole entries), two and
    # four query tokens with rows that see no key, an empty entry, and long
    # entries split across clusters.
    (117, 300, 1, 16, list(W.uniform_int(117, W.TENSOR_SEQLENS, 300, 1, 200)), 0),
    (118, 4, 2, 8, [1, 64, 65, 20000], 1),
    (119, 4, 4, 4, [0, 2, 900, 25000], 1),
    (124, 2, 1, 16, [20000, 9000], 0),
    # fewer rows than the narrow kernel's 16: one head, and four heads
    (127, 3, 1, 1, [9000, 70, 30000], 1),
    (128, 2, 1, 4, [20000, 15000], 0),
    # 17 to 32 rows: the narrow kernel's 32-row form (two speculative tokens
    # of 16 heads with a row that sees no key, 32 heads, 3 tokens x 8 heads,
    # many short entries)
    (129, 4, 2, 16, [1, 700, 5000, 20000], 1),
    (130, 3, 1, 32, [30000, 64, 129], 0),
    (131, 2, 3, 8, [25000, 17], 1),
    (132, 200, 2, 16, list(W.uniform_int(132, W.TENSOR_SEQLENS, 200, 1, 300)), 0),
]


# The exact result of this case holds values of magnitude 4 to 4.6, where
# bf16 values are 2^-5 apart: rounded to bf16, the fp64 oracle's own output is
# 1.40e-2 from itself (tests/test_output_format.py), so no bf16 output can
# meet 1e-2 there.  Its fp32 output is held to the bar like every other case,
# and its bf16 output must be that fp32 output rounded to nearest even.
BF16_UNREPRESENTABLE = {112}


@pytest.mark.parametrize("case", SMALL, ids=lambda c: f"s{c[0]}_b{c[1]}_sq{c[2]}_h{c[3]}")
def test_small_parity(torch_cuda, case, oracle_mod):
    seed, B, s_q, h_q, seqlens, extra = case
    inp = W.make_inputs(seed, B, s_q, h_q, seqlens, extra_pages=extra)
    ref_o, ref_l = oracle_mod.mla_decode(inp)
    out32, lse32, _ = run_gpu(torch_cuda, inp, out_f32=True)
    eo, el = assert_parity(out32, lse32, ref_o, ref_l, f"case {seed} fp32 out")
    out16, lse16, _ = run_gpu(torch_cuda, inp)
    assert np.array_equal(lse16, lse32), f"case {seed}: lse differs between the two outputs"
    assert_bf16_is_rounded_f32(out16, out32, f"case {seed}")
    if seed not in BF16_UNREPRESENTABLE:
        assert_parity(out16, lse16, ref_o, ref_l, f"case {seed} bf16 out")


def test_narrow_cases_take_the_narrow_kernel(torch_cuda):
    """The cases meant for the narrow kernel do run it (and the small ones
    with few rows stay on the general kernel)."""
    nc = libmla.mla_num_clusters(0)
    for seed, B, s_q, h_q, seqlens, extra in SMALL:
        inp = W.make_inputs(seed, B, s_q, h_q, seqlens, extra_pages=extra)
        kind = libmla.mla_decode_kernel_kind(B, s_q, h_q, int(inp.block_table.shape[1]))
        want = s_q * h_q <= 32 and B * inp.block_table.shape[1] > 4 * nc
        assert kind == (1 if want else 0), (seed, kind)
        if seed in (117, 118, 119, 124, 127, 128, 129, 130, 131, 132):
            assert kind == 1, seed


@pytest.mark.parametrize("case", [c for c in SMALL if c[0] in (104, 106, 113, 115, 117, 124)],
                         ids=lambda c: f"s{c[0]}")
def test_split_route_matches(torch_cuda, case, oracle_mod):
    """mla_decode_attend (the main kernel: whole entries written out, split
    partials left in the workspace) followed by mla_decode_combine (the LSE
    merge) is mla_decode in two calls: the same result, bit for bit, and
    the oracle's within the bar."""
    seed, B, s_q, h_q, seqlens, extra = case
    inp = W.make_inputs(seed, B, s_q, h_q, seqlens, extra_pages=extra)
    ref_o, ref_l = oracle_mod.mla_decode(inp)
    fused_o, fused_l, _ = run_gpu(torch_cuda, inp)
    d = to_device(torch_cuda, inp)
    out = torch_cuda.full((B, s_q, h_q, 512), float("nan"), dtype=torch_cuda.bfloat16, device="cuda")
    lse = torch_cuda.full((B, h_q, s_q), float("nan"), dtype=torch_cuda.float32, device="cuda")
    meta, ws = libmla.alloc_plan_and_workspace(B, s_q, h_q, 0)
    ws.fill_(float("nan"))
    libmla.mla_decode_plan(d["sl"], s_q, h_q, meta)
    libmla.mla_decode_attend(d["q"], d["kv"], d["bt"], d["sl"], meta, out, lse,
                             inp.softmax_scale, ws)
    libmla.mla_decode_combine(B, s_q, h_q, meta, out, lse, ws)
    assert libmla.mla_check_device_error() == 0
    split_o, split_l = out.float().cpu().numpy(), lse.cpu().numpy()
    assert_parity(split_o, split_l, ref_o, ref_l, f"case {seed} split route")
    assert np.array_equal(split_o, fused_o) and np.array_equal(split_l, fused_l)


def _sample_rows(w, inp, n, seed):
    rng = np.random.default_rng(seed)
    rows = np.stack([rng.integers(0, w.batch, n), rng.integers(0, w.s_q, n),
                     rng.integers(0, w.h_q, n)], axis=1)
    # always include the corners
    corners = np.array([[0, 0, 0], [w.batch - 1, w.s_q - 1, w.h_q - 1]])
    return np.concatenate([corners, rows]).astype(np.int32)


@pytest.mark.parametrize("name", list(W.WORKLOADS))
def test_workload_parity(torch_cuda, name, oracle_mod):
    """The five decode workloads at full size through the same C-ABI call the
    benchmark times: every element for the cheap ones, 400 sampled rows of
    the 602-GFLOP two-token workload."""
    w = W.WORKLOADS[name]
    inp = w.make()
    out, lse, _ = run_gpu(torch_cuda, inp)
    if w.flops() < 1e11:
        ref_o, ref_l = oracle_mod.mla_decode(inp)
        assert_parity(out, lse, ref_o, ref_l, name)
    else:
        rows = _sample_rows(w, inp, 400, 5)
        ref_o, ref_l = oracle_mod.mla_decode_rows(inp, rows)
        got_o = out[rows[:, 0], rows[:, 1], rows[:, 2]]
        got_l = lse[rows[:, 0], rows[:, 2], rows[:, 1]]
        assert_parity(got_o, got_l, ref_o, ref_l, name)
        assert not np.isnan(out).any() and not np.isnan(lse).any()


def test_device_plan_matches_host_plan(torch_cuda):
    for seqlens, s_q, h_q in [([4096] * 16, 1, 128), ([0, 1, 65, 7000, 3], 2, 128),
                              (list(W.uniform_int(2, W.TENSOR_SEQLENS, 64, 1, 8192)), 1, 128),
                              ([65536] * 8, 1, 16)]:
        sl = np.asarray(seqlens, dtype=np.int32)
        nc = libmla.mla_num_clusters(0)
        host = libmla.mla_decode_plan_host(sl, s_q, h_q, nc)
        meta, _ = libmla.alloc_plan_and_workspace(len(sl), s_q, h_q, 0)
        meta.zero_()
        libmla.mla_decode_plan(torch_cuda.from_numpy(sl).cuda(), s_q, h_q, meta)
        dev = meta.cpu().numpy()[: host.shape[0]]
        n = libmla.mla_plan_size_for_clusters(len(sl), s_q, h_q, nc) // 4
        assert np.array_equal(dev[:n], host[:n])
        assert libmla.mla_check_device_error() == 0


def test_deterministic_and_relabel_invariant(torch_cuda):
    inp = W.make_inputs(120, 3, 2, 128, [900, 64, 2500], extra_pages=3)
    o1, l1, _ = run_gpu(torch_cuda, inp)
    o2, l2, _ = run_gpu(torch_cuda, inp)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)
    relabel = W.permutation(77, 3, inp.num_pages)
    kv = np.empty_like(inp.kv_cache)
    kv[relabel] = inp.kv_cache
    moved = W.DecodeInputs(q=inp.q, kv_cache=kv, block_table=relabel[inp.block_table],
                           cache_seqlens=inp.cache_seqlens, s_q=2, h_q=128)
    o3, l3, _ = run_gpu(torch_cuda, moved)
    assert np.array_equal(o1, o3) and np.array_equal(l1, l3)


@pytest.mark.parametrize("s_q,h_q,seqlens", [(1, 16, [12000, 7000]), (2, 8, [12000, 7000]),
                                             (2, 16, [12000, 7000]),
                                             (1, 16, [3000, 1700]), (1, 128, [3000, 1700]),
                                             (2, 64, [3000, 1700])])
def test_growing_scores_rescale(torch_cuda, oracle_mod, s_q, h_q, seqlens):
    """Scores that grow along the sequence (a rotary dim of every key set to
    a ramp, q's matching dim to 2) move the running max by more than the lazy
    rescale threshold many times per entry: O and the sums are rescaled on
    the GPU (the narrow kernel, 16- and 32-row forms, for the first three;
    the general one for the rest), and the result must still match the
    oracle."""
    inp = W.make_inputs(125, 2, s_q, h_q, seqlens, poison=False)
    d = W.D_QK - 1
    for b in range(inp.batch):
        L = int(inp.cache_seqlens[b])
        t = np.arange(L)
        inp.kv_cache[inp.block_table[b, t // 64], t % 64, 0, d] = W.float32_to_bf16_bits(
            t.astype(np.float32) * np.float32(0.05))
    inp.q[..., d] = W.float32_to_bf16_bits(np.float32([2.0]))[0]
    ref_o, ref_l = oracle_mod.mla_decode(inp)
    out, lse, _ = run_gpu(torch_cuda, inp, out_f32=True)
    assert_parity(out, lse, ref_o, ref_l, f"ramp s_q={s_q} h_q={h_q}")


def test_shift_invariance_on_gpu(torch_cuda):
    """A common logit shift (a rotary dim set to 2 in every key, q's matching
    dim moved by 0.5) leaves out unchanged and moves lse by scale * 1."""
    inp = W.make_inputs(121, 2, 1, 128, [700, 300], poison=False)
    d = W.D_QK - 1
    inp.kv_cache[..., d] = W.float32_to_bf16_bits(np.float32([2.0]))[0]
    inp.q[..., d] = 0
    o0, l0, _ = run_gpu(torch_cuda, inp)
    inp.q[..., d] = W.float32_to_bf16_bits(np.float32([0.5]))[0]
    o1, l1, _ = run_gpu(torch_cuda, inp)
    assert float(np.abs(o1 - o0).max()) <= OUT_TOL
    assert float(np.abs((l1 - l0) - W.SOFTMAX_SCALE).max()) <= LSE_TOL


def test_bad_page_index_is_reported_not_faulted(torch_cuda):
    inp = W.make_inputs(122, 2, 1, 16, [100, 200])
    d = to_device(torch_cuda, inp)
    d["bt"][1, 1] = inp.num_pages + 5          # out of range: clamped, flagged
    _, _, _ = run_gpu(torch_cuda, inp, d, check_err=False)
    # run_gpu already consumed the error word; run again and read it here
    out = torch_cuda.empty((2, 1, 16, 512), dtype=torch_cuda.bfloat16, device="cuda")
    lse = torch_cuda.empty((2, 16, 1), dtype=torch_cuda.float32, device="cuda")
    meta, ws = libmla.alloc_plan_and_workspace(2, 1, 16, 0)
    libmla.mla_decode_plan(d["sl"], 1, 16, meta)
    libmla.mla_decode(d["q"], d["kv"], d["bt"], d["sl"], meta, out, lse, inp.softmax_scale, ws)
    assert libmla.mla_check_device_error() == libmla.MLA_ERR_DEVICE_BOUNDS
    assert libmla.mla_check_device_error() == 0     # the word is cleared


def test_mismatched_plan_is_reported(torch_cuda):
    inp = W.make_inputs(123, 2, 1, 64, [100, 200])
    d = to_device(torch_cuda, inp)
    meta, ws = libmla.alloc_plan_and_workspace(2, 1, 64, 0)
    libmla.mla_decode_plan(d["sl"], 1, 32, meta)           # planned for h_q = 32
    out = torch_cuda.empty((2, 1, 64, 512), dtype=torch_cuda.bfloat16, device="cuda")
    lse = torch_cuda.empty((2, 64, 1), dtype=torch_cuda.float32, device="cuda")
    libmla.mla_decode(d["q"], d["kv"], d["bt"], d["sl"], meta, out, lse, inp.softmax_scale, ws)
    assert libmla.mla_check_device_error() == libmla.MLA_ERR_PLAN


def test_plan_covers_all_pages_on_device(torch_cuda):
    """The device plan for the ragged workload partitions every page."""
    w = W.WORKLOADS["ragged_b64_h128"]
    sl = w.seqlens()
    meta, _ = libmla.alloc_plan_and_workspace(w.batch, 1, 128, 0)
    libmla.mla_decode_plan(torch_cuda.from_numpy(sl).cuda(), 1, 128, meta)
    plan = plan_model.decode(meta.cpu().numpy())
    seen = set()
    for c in range(plan["gt"]):
        for (b, pb, pe, _) in plan_model.segments(plan, c):
            for p in range(pb, pe):
                assert (b, p) not in seen
                seen.add((b, p))
    assert len(seen) == sum((int(L) + 63) // 64 for L in sl)


def test_bounded_wait_times_out_and_context_survives(torch_cuda, oracle_mod):
    """A wait nothing satisfies gives up (about 2 s), reports
    MLA_ERR_DEVICE_TIMEOUT, and the next decode on the same context is
    correct."""
    libmla.mla_check_device_error()      # start from a clear error word
    libmla.mla_selftest_wait_timeout()
    assert libmla.mla_check_device_error() == libmla.MLA_ERR_DEVICE_TIMEOUT
    assert libmla.mla_check_device_error() == 0          # read and cleared
    inp = W.make_inputs(121, 2, 1, 128, [200, 64], extra_pages=1)
    out, lse, _ = run_gpu(torch_cuda, inp)
    ref_o, ref_l = oracle_mod.mla_decode(inp)
    assert_parity(out, lse, ref_o, ref_l, "after timeout")
