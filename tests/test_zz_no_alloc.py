"""mla_decode_noalloc against mla_decode (needs a GB300).

Some callers cannot allocate device memory: frameworks whose own allocator
owns every byte on the GPU and does not let an operator call cudaMalloc, and
serving loops that must stay out of the CUDA allocator.  mla_decode_noalloc
serves them by keeping the split-KV partials in a static array inside the
library.  This test calls it twice in a row through the C ABI, on workloads
whose batch entries are split over several clusters (so the partials, and
therefore the static array, are really used), and checks each result against
the workspace-taking mla_decode within the parity tolerances of the other GPU
tests.  It lives in its own file, collected last, and passes both alone in a
fresh process and after the rest of the suite.
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


def _device_inputs(torch, inp):
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    return (t(inp.q.view(np.int16)).view(torch.bfloat16),
            t(inp.kv_cache.view(np.int16)).view(torch.bfloat16),
            t(inp.block_table), t(inp.cache_seqlens))


@pytest.mark.parametrize("seed,batch,s_q,h_q,seqlens", [
    (201, 4, 1, 128, [3000, 2500, 4096, 100]),
    (202, 3, 2, 64, [5000, 1, 777]),
])
def test_noalloc_matches_workspace_entry_point(torch_cuda, seed, batch, s_q, h_q, seqlens):
    torch = torch_cuda
    inp = W.make_inputs(seed, batch, s_q, h_q, seqlens, extra_pages=1)
    q, kv, bt, sl = _device_inputs(torch, inp)
    meta, ws = libmla.alloc_plan_and_workspace(batch, s_q, h_q, 0)
    libmla.mla_decode_plan(sl, s_q, h_q, meta)
    ref_out = torch.empty((batch, s_q, h_q, 512), dtype=torch.bfloat16, device="cuda")
    ref_lse = torch.empty((batch, h_q, s_q), dtype=torch.float32, device="cuda")
    libmla.mla_decode(q, kv, bt, sl, meta, ref_out, ref_lse, inp.softmax_scale, ws)
    assert libmla.mla_check_device_error() == 0
    # the plan really splits entries over clusters, so the scratch is used
    plan = plan_model.decode(meta.cpu().numpy())
    assert (plan["items"][:, 1] >= 2).any()
    ro = ref_out.float().cpu().numpy()
    rl = ref_lse.cpu().numpy()
    for call in range(2):
        out = torch.full_like(ref_out, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        libmla.mla_decode_noalloc(q, kv, bt, sl, meta, out, lse, inp.softmax_scale)
        assert libmla.mla_check_device_error() == 0
        o = out.float().cpu().numpy()
        l = lse.cpu().numpy()
        assert not np.isnan(o).any() and not np.isnan(l).any(), f"call {call}: NaN"
        assert np.array_equal(np.isneginf(l), np.isneginf(rl))
        assert float(np.abs(o - ro).max()) <= OUT_TOL, f"call {call}: out"
        fin = ~np.isneginf(rl)
        assert float(np.abs(l[fin] - rl[fin]).max()) <= LSE_TOL, f"call {call}: lse"
