"""Split-KV planner invariants, via the host planner (CPU only).

The device planner is checked bit for bit against this one in the GPU tests.
"""
import numpy as np
import pytest

import plan_model
from mla_decode_attention_07_gb300 import libmla
from mla_decode_attention_07_gb300 import workloads as W


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    __graft_entry__.build_library()


CASES = [
    ([256], 1, 16, 76),
    ([4096] * 16, 1, 128, 76),
    ([8192] * 132, 2, 128, 76),
    ([65536] * 8, 1, 16, 76),
    (list(W.uniform_int(2, W.TENSOR_SEQLENS, 64, 1, 8192)), 1, 128, 76),
    ([0, 1, 63, 64, 65, 0, 200, 1000], 2, 64, 76),
    ([1], 1, 1, 76),
    ([0, 0, 0], 1, 128, 76),
    (list(W.uniform_int(7, 9, 300, 0, 3000)), 1, 128, 75),
    ([5000, 3, 70000, 64], 1, 128, 5),
    ([100] * 20, 3, 100, 74),
    (list(W.uniform_int(112, W.TENSOR_SEQLENS, 300, 1, 64)), 1, 128, 76),
]


@pytest.mark.parametrize("seqlens,s_q,h_q,nc", CASES)
def test_plan_partition(seqlens, s_q, h_q, nc):
    sl = np.asarray(seqlens, dtype=np.int32)
    meta = libmla.mla_decode_plan_host(sl, s_q, h_q, nc)
    plan = plan_model.decode(meta)
    hdr = plan["header"]
    B = len(sl)
    T = (s_q * h_q + 127) // 128
    assert hdr[plan_model.H_MAGIC] == plan_model.MAGIC
    assert (hdr[plan_model.H_BATCH], hdr[plan_model.H_SQ], hdr[plan_model.H_HQ]) == (B, s_q, h_q)
    assert plan["tiles"] == T and plan["gt"] == nc // T
    assert hdr[plan_model.H_NCLUSTERS] == nc
    pages = [(int(L) + 63) // 64 if L > 0 else 0 for L in sl]
    assert [int(x) for x in plan["items"][:, 0]] == pages

    covered = {}
    seg_of = {b: [] for b in range(B)}
    for c in range(plan["gt"]):
        segs = plan_model.segments(plan, c)
        if c >= plan["gused"]:
            assert not segs
        for (b, pb, pe, sidx) in segs:
            assert 0 <= pb < pe <= pages[b]
            for p in range(pb, pe):
                assert (b, p) not in covered, "page processed twice"
                covered[(b, p)] = c
            seg_of[b].append((c, pb, pe, sidx))
    assert set(covered) == {(b, p) for b in range(B) for p in range(pages[b])}

    stotal = 0
    for b in range(B):
        ns = int(plan["items"][b][1])
        segs = seg_of[b]
        assert ns == len(segs)
        if pages[b] == 0:
            assert ns == 0
            continue
        # clusters of one entry are consecutive, pages contiguous and in order,
        # split indices 0..ns-1
        cs = [s[0] for s in segs]
        assert cs == list(range(cs[0], cs[0] + ns))
        assert segs[0][1] == 0 and segs[-1][2] == pages[b]
        for k in range(1, ns):
            assert segs[k][1] == segs[k - 1][2]
        assert [s[3] for s in segs] == list(range(ns))
        if ns >= 2:
            assert int(plan["items"][b][2]) == stotal
            stotal += ns
    assert plan["stotal"] == stotal <= 2 * plan["gt"]

    # balance: cluster loads within a few units of an equal share, where an
    # entry costs its pages plus the plan's per-entry overhead (charged to the
    # cluster that starts the entry)
    ovh = int(plan["header"][plan_model.H_OVH])
    assert ovh >= 0
    load = {}
    for (b, p), c in covered.items():
        load[c] = load.get(c, 0) + 1
    for b in range(B):
        for (c, pb, pe, s) in seg_of[b]:
            if pb == 0:
                load[c] += ovh
    if load:
        total = sum(pages) + ovh * sum(1 for p in pages if p)
        quota = -(-total // max(1, plan["gused"]))
        assert max(load.values()) <= quota + ovh + 1


def test_plan_rejects_bad_args():
    with pytest.raises(libmla.MlaError):
        libmla.mla_decode_plan_host(np.array([10], np.int32), 1, 129, 76)
    with pytest.raises(libmla.MlaError):
        libmla.mla_decode_plan_host(np.array([10], np.int32), 9, 16, 76)
    assert libmla.mla_plan_size_for_clusters(4, 2, 128, 1) == 0   # 2 tiles need >= 2 clusters
