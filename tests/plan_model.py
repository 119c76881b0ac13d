"""Reads the split-KV tile metadata the way the decode kernel walks it.

The layout mirrors the plan header, cluster table, item table and unit
starts written by the planner; this module only decodes it so the tests can
check the partition (it computes nothing of its own).
"""
from __future__ import annotations

import numpy as np

H_WORDS = 16
H_MAGIC, H_BATCH, H_SQ, H_HQ, H_TILES, H_GT, H_GUSED, H_STOTAL, H_OVH, H_NCLUSTERS = range(10)
MAGIC = 0x4D4C4131
CLUSTER_WORDS = 8
ITEM_WORDS = 4


def decode(meta: np.ndarray) -> dict:
    m = np.asarray(meta).view(np.int32)
    hdr = m[:H_WORDS]
    gt, batch = int(hdr[H_GT]), int(hdr[H_BATCH])
    clus = m[H_WORDS:H_WORDS + gt * CLUSTER_WORDS].reshape(gt, CLUSTER_WORDS)
    off_items = H_WORDS + gt * CLUSTER_WORDS
    items = m[off_items:off_items + batch * ITEM_WORDS].reshape(batch, ITEM_WORDS)
    return dict(header=hdr, clusters=clus, items=items, gt=gt, batch=batch,
                tiles=int(hdr[H_TILES]), gused=int(hdr[H_GUSED]), stotal=int(hdr[H_STOTAL]))


def segments(plan: dict, c: int):
    """(b, page_begin, page_end, split_index) in the order cluster c runs them."""
    b0, p0, b1, p1, split0 = (int(v) for v in plan["clusters"][c][:5])
    items = plan["items"]
    out = []
    b, p = b0, p0
    while b < b1 or (b == b1 and p < p1):
        P = int(items[b][0])
        pe = p1 if b == b1 else P
        if p < pe:
            out.append((b, p, pe, split0 if not out else 0))
        b, p = b + 1, 0
    return out
