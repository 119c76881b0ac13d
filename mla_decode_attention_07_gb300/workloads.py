"""Seeded synthetic inputs for paged MLA decode.

This module only draws numbers and lays them out: it holds none of the
attention arithmetic, so both the CUDA path and the CPU oracle can consume
the same bits without sharing any of the method's code.

Random source: SplitMix64 (Steele, Lea & Flood, "Fast splittable
pseudorandom number generators", OOPSLA 2014), used in counter form: output k
of the stream with start value ``s`` is ``mix(s + (k + 1) * GAMMA)`` mod 2**64.
Each tensor has its own stream, started at ``seed ^ TENSOR_ID``.

Normals: Box-Muller on two 53-bit uniforms in (0, 1], computed in float64,
rounded to float32 and then to bfloat16 with round-to-nearest-even.

Shapes (DeepSeek-style MLA decode over a paged latent cache):
  q            [B, s_q, h_q, 576]      bf16 (uint16 bits)
  kv_cache     [num_pages, 64, 1, 576] bf16 (uint16 bits)
  block_table  [B, max_pages]          int32
  cache_seqlens[B]                     int32
Sparse decode adds, with s_q = 1:
  indices      [B, topk]               int32 token positions, -1 past counts[b]
  counts       [B]                     int32 selected positions per entry
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

D_QK = 576          # 512 latent + 64 rope dims per cache row
D_V = 512           # values are the first 512 dims of the same row
PAGE = 64           # tokens per KV page
SOFTMAX_SCALE = 192.0 ** -0.5

GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

TENSOR_Q = 0x51
TENSOR_KV = 0x4B56
TENSOR_SEQLENS = 0x5345
TENSOR_PERM = 0x5045
TENSOR_IDX = 0x4958        # sparse: token positions selected per batch entry
TENSOR_POOL = 0x504C       # sparse: block-table draws into a shared page pool

BF16_NAN = np.uint16(0x7FC0)


def splitmix64(start: int, first: int, count: int) -> np.ndarray:
    """Outputs ``first .. first+count-1`` of the SplitMix64 stream at ``start``."""
    k = np.arange(first + 1, first + count + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = np.uint64(start & 0xFFFFFFFFFFFFFFFF) + k * GAMMA
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def _uniform01(z: np.ndarray) -> np.ndarray:
    # 53 high bits -> (0, 1]
    return ((z >> np.uint64(11)).astype(np.float64) + 1.0) * (2.0 ** -53)


def float32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (nearest-even) and return the bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    with np.errstate(over="ignore"):
        r = (u + bias) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_float32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _normal_chunk(start: int, first_pair: int, pairs: int, out: np.ndarray, n: int) -> None:
    z = splitmix64(start, 2 * first_pair, 2 * pairs)
    u1 = _uniform01(z[0::2])
    u2 = _uniform01(z[1::2])
    r = np.sqrt(-2.0 * np.log(u1))
    th = 2.0 * math.pi * u2
    vals = np.empty(2 * pairs, dtype=np.float64)
    vals[0::2] = r * np.cos(th)
    vals[1::2] = r * np.sin(th)
    lo = 2 * first_pair
    hi = min(n, lo + 2 * pairs)
    out[lo:hi] = float32_to_bf16_bits(vals[: hi - lo].astype(np.float32))


def normal_bf16(seed: int, tensor_id: int, n: int, chunk: int = 1 << 20) -> np.ndarray:
    """``n`` N(0,1) samples rounded to bf16 bits, deterministic in (seed, tensor_id).

    Large requests are cut into fixed chunks that threads fill independently;
    the values do not depend on the chunking or the thread count.
    """
    start = (seed ^ tensor_id) & 0xFFFFFFFFFFFFFFFF
    out = np.empty(n, dtype=np.uint16)
    pairs_total = (n + 1) // 2
    jobs = [(p0, min(chunk, pairs_total - p0)) for p0 in range(0, pairs_total, chunk)]
    if len(jobs) <= 1:
        for p0, m in jobs:
            _normal_chunk(start, p0, m, out, n)
        return out
    import concurrent.futures as cf
    import os
    with cf.ThreadPoolExecutor(max_workers=min(len(jobs), os.cpu_count() or 1)) as ex:
        list(ex.map(lambda j: _normal_chunk(start, j[0], j[1], out, n), jobs))
    return out


def uniform_int(seed: int, tensor_id: int, n: int, lo: int, hi: int) -> np.ndarray:
    """``n`` integers uniform in [lo, hi] (inclusive)."""
    span = hi - lo + 1
    z = splitmix64((seed ^ tensor_id) & 0xFFFFFFFFFFFFFFFF, 0, n)
    return (lo + (z % np.uint64(span)).astype(np.int64)).astype(np.int32)


def permutation(seed: int, tensor_id: int, n: int) -> np.ndarray:
    """A uniformly random permutation of range(n): argsort of 64-bit keys."""
    z = splitmix64((seed ^ tensor_id) & 0xFFFFFFFFFFFFFFFF, 0, n)
    return np.argsort(z, kind="stable").astype(np.int32)


@dataclasses.dataclass
class DecodeInputs:
    q: np.ndarray            # uint16 [B, s_q, h_q, 576]
    kv_cache: np.ndarray     # uint16 [num_pages, 64, 1, 576]
    block_table: np.ndarray  # int32 [B, max_pages]
    cache_seqlens: np.ndarray  # int32 [B]
    s_q: int
    h_q: int
    softmax_scale: float = SOFTMAX_SCALE

    @property
    def batch(self) -> int:
        return int(self.cache_seqlens.shape[0])

    @property
    def num_pages(self) -> int:
        return int(self.kv_cache.shape[0])

    @property
    def max_pages(self) -> int:
        return int(self.block_table.shape[1])


def make_inputs(seed: int, batch: int, s_q: int, h_q: int, seqlens, *,
                extra_pages: int = 0, poison: bool = True,
                q_zero: bool = False) -> DecodeInputs:
    """Seeded decode inputs.

    ``seqlens`` is a sequence of ints (one per batch entry).  The pool holds
    exactly ``sum(ceil(L/64))`` live pages plus ``extra_pages`` decoy pages,
    all in a random order.  With ``poison`` the unused tail slots of every last
    page, the decoy pages and the unused block-table entries (which point at a
    decoy page, or at page 0 when there is none) hold NaN-poisoned data, so a
    kernel that reads anything it should not shows NaN in its output.
    """
    seqlens = np.asarray(seqlens, dtype=np.int32).reshape(batch)
    if np.any(seqlens < 0):
        raise ValueError("sequence lengths must be >= 0")
    pages_per = [(int(L) + PAGE - 1) // PAGE for L in seqlens]
    live = int(sum(pages_per))
    num_pages = live + int(extra_pages)
    if num_pages == 0:
        num_pages = 1
    max_pages = max(1, max(pages_per) if pages_per else 1)

    perm = permutation(seed, TENSOR_PERM, num_pages)
    block_table = np.empty((batch, max_pages), dtype=np.int32)
    decoy = int(perm[live]) if num_pages > live else int(perm[0])
    block_table[:] = decoy
    off = 0
    for b, np_b in enumerate(pages_per):
        block_table[b, :np_b] = perm[off:off + np_b]
        off += np_b

    kv = normal_bf16(seed, TENSOR_KV, num_pages * PAGE * D_QK).reshape(num_pages, PAGE, 1, D_QK)
    q = normal_bf16(seed, TENSOR_Q, batch * s_q * h_q * D_QK).reshape(batch, s_q, h_q, D_QK)
    if q_zero:
        q[:] = 0
    if poison:
        for b, np_b in enumerate(pages_per):
            L = int(seqlens[b])
            if np_b and L % PAGE:
                kv[block_table[b, np_b - 1], L % PAGE:] = BF16_NAN
        for p in perm[live:]:
            kv[int(p)] = BF16_NAN
    return DecodeInputs(q=q, kv_cache=kv, block_table=block_table,
                        cache_seqlens=seqlens, s_q=s_q, h_q=h_q)


@dataclasses.dataclass(frozen=True)
class Workload:
    """One named decode workload: shapes plus the seeded recipe."""
    name: str
    batch: int
    s_q: int
    h_q: int
    seqlen: int | None      # uniform length, or None for seeded ragged lengths
    seqlen_max: int = 0     # upper bound of the ragged draw
    seed: int = 0

    def seqlens(self) -> np.ndarray:
        if self.seqlen is not None:
            return np.full(self.batch, self.seqlen, dtype=np.int32)
        return uniform_int(self.seed, TENSOR_SEQLENS, self.batch, 1, self.seqlen_max)

    def make(self, **kw) -> DecodeInputs:
        return make_inputs(self.seed, self.batch, self.s_q, self.h_q, self.seqlens(), **kw)

    def visible_keys(self) -> int:
        """Sum over (batch, query token) of visible keys (bottom-right causal)."""
        L = self.seqlens().astype(np.int64)
        tot = 0
        for i in range(self.s_q):
            tot += int(np.maximum(L - self.s_q + 1 + i, 0).sum())
        return tot

    def flops(self) -> float:
        """Algorithmic flops: 2 * (576 + 512) per (head, visible key)."""
        return 2.0 * (D_QK + D_V) * self.h_q * self.visible_keys()

    def bytes(self) -> float:
        """Algorithmic bytes: each live cache row once, plus q, out and lse."""
        L = self.seqlens().astype(np.int64)
        kv = int(L.sum()) * D_QK * 2
        rows = self.batch * self.s_q * self.h_q
        return float(kv + rows * D_QK * 2 + rows * D_V * 2 + rows * 4)


# The five decode workloads: tiny, large-batch 128-head, ragged, two-token
# speculative (causal inside the two query tokens) and long-context 16-head.
WORKLOADS = {
    "tiny": Workload("tiny", batch=1, s_q=1, h_q=16, seqlen=256, seed=0),
    "b16_h128_l4096": Workload("b16_h128_l4096", batch=16, s_q=1, h_q=128, seqlen=4096, seed=1),
    "ragged_b64_h128": Workload("ragged_b64_h128", batch=64, s_q=1, h_q=128, seqlen=None,
                                seqlen_max=8192, seed=2),
    "spec_b132_sq2_h128_l8192": Workload("spec_b132_sq2_h128_l8192", batch=132, s_q=2, h_q=128,
                                         seqlen=8192, seed=3),
    "long_b8_h16_l65536": Workload("long_b8_h16_l65536", batch=8, s_q=1, h_q=16, seqlen=65536,
                                   seed=4),
}


@dataclasses.dataclass
class SparseInputs:
    """Sparse decode inputs: a paged cache (``base``, s_q = 1) plus, per batch
    entry, the list of token positions its query attends to."""
    base: DecodeInputs
    indices: np.ndarray      # int32 [B, topk]; entries past counts[b] are -1
    counts: np.ndarray       # int32 [B]

    @property
    def topk(self) -> int:
        return int(self.indices.shape[1])


def draw_indices(seed: int, seqlens, topk: int, counts=None, *,
                 repeats: bool = False) -> tuple[np.ndarray, np.ndarray]:
    """Per entry b, ``counts[b]`` token positions in [0, L_b) (default
    min(topk, L_b)) in random order: distinct (a random subset), or with
    ``repeats`` drawn independently.  Slots past counts[b] hold -1."""
    seqlens = np.asarray(seqlens, dtype=np.int64)
    B = seqlens.shape[0]
    if counts is None:
        counts = np.minimum(seqlens, topk)
    counts = np.asarray(counts, dtype=np.int32).reshape(B)
    idx = np.full((B, topk), -1, dtype=np.int32)
    for b in range(B):
        L, c = int(seqlens[b]), int(counts[b])
        if c == 0:
            continue
        if c > topk or (c > L and not repeats) or L == 0:
            raise ValueError("count out of range")
        sb = (seed * 1000003 + b) & 0xFFFFFFFFFFFFFFFF
        if repeats:
            z = splitmix64(sb ^ TENSOR_IDX, 0, c)
            idx[b, :c] = (z % np.uint64(L)).astype(np.int64)
        else:
            z = splitmix64(sb ^ TENSOR_IDX, 0, L)
            idx[b, :c] = np.argsort(z, kind="stable")[:c]
    return idx, counts


def make_sparse_inputs(seed: int, batch: int, h_q: int, seqlens, topk: int, counts=None, *,
                       repeats: bool = False, pool_pages: int | None = None,
                       poison: bool = True) -> SparseInputs:
    """Seeded sparse decode inputs (one query token per entry).

    Without ``pool_pages`` the cache is ``make_inputs``' (every live page
    once, NaN-poisoned tails and decoys).  With it, the cache is a shared
    pool of that many pages and every block-table entry is a uniform draw
    from the pool, so long contexts need not be stored in full (pages repeat
    across and within entries, as with a shared prefix)."""
    seqlens = np.asarray(seqlens, dtype=np.int32).reshape(batch)
    if pool_pages is None:
        base = make_inputs(seed, batch, 1, h_q, seqlens, extra_pages=2, poison=poison)
    else:
        max_pages = max(1, max((int(L) + PAGE - 1) // PAGE for L in seqlens))
        bt = uniform_int(seed, TENSOR_POOL, batch * max_pages, 0, pool_pages - 1)
        kv = normal_bf16(seed, TENSOR_KV, pool_pages * PAGE * D_QK).reshape(pool_pages, PAGE, 1,
                                                                           D_QK)
        q = normal_bf16(seed, TENSOR_Q, batch * h_q * D_QK).reshape(batch, 1, h_q, D_QK)
        base = DecodeInputs(q=q, kv_cache=kv, block_table=bt.reshape(batch, max_pages),
                            cache_seqlens=seqlens, s_q=1, h_q=h_q)
    idx, cnt = draw_indices(seed, seqlens, topk, counts, repeats=repeats)
    return SparseInputs(base=base, indices=idx, counts=cnt)


@dataclasses.dataclass(frozen=True)
class SparseWorkload:
    """One named sparse decode workload (s_q = 1)."""
    name: str
    batch: int
    h_q: int
    seqlen: int
    topk: int
    pool_pages: int
    seed: int = 0

    def make(self) -> SparseInputs:
        return make_sparse_inputs(self.seed, self.batch, self.h_q,
                                  np.full(self.batch, self.seqlen, dtype=np.int32), self.topk,
                                  pool_pages=self.pool_pages)

    def keys(self) -> int:
        return self.batch * min(self.topk, self.seqlen)

    def flops(self) -> float:
        """2 * (576 + 512) per (head, selected key)."""
        return 2.0 * (D_QK + D_V) * self.h_q * self.keys()

    def bytes(self) -> float:
        """Each selected cache row once, plus q, out, lse and the indices."""
        rows = self.batch * self.h_q
        return float(self.keys() * (D_QK * 2 + 4) + rows * D_QK * 2 + rows * D_V * 2 + rows * 4)


# Sparse decode at 128K context: 2048 selected positions per entry, 128
# heads; the cache is a 604 MB pool of 8192 pages shared by the 64 entries'
# block tables.
SPARSE_WORKLOADS = {
    "sparse_b64_h128_l131072_k2048": SparseWorkload("sparse_b64_h128_l131072_k2048", batch=64,
                                                    h_q=128, seqlen=131072, topk=2048,
                                                    pool_pages=8192, seed=5),
}


# ---------------------------------------------------------------------------
# The steps before the decode call (DeepSeek MLA): the new tokens' cache rows
# and the query parts the absorption contracts, and the tensor-core GEMM's
# factors.  Only numbers are drawn here; the arithmetic is elsewhere.
D_NOPE = 128        # per-head query dims contracted with W_UK
D_ROPE = 64         # per-head rotary query dims (the last 64 of the 576)
D_C = 512           # latent dims

TENSOR_KV_NEW = 0x4E57
TENSOR_Q_NOPE = 0x514E
TENSOR_Q_ROPE = 0x5152
TENSOR_W_UK = 0x574B
TENSOR_GEMM_A = 0x4741
TENSOR_GEMM_B = 0x4742


def normal_f16(seed: int, tensor_id: int, n: int) -> np.ndarray:
    """``n`` N(0,1) samples (the same Box-Muller stream as normal_bf16)
    rounded to float32, then to IEEE binary16 with round-to-nearest-even."""
    start = (seed ^ tensor_id) & 0xFFFFFFFFFFFFFFFF
    pairs = (n + 1) // 2
    z = splitmix64(start, 0, 2 * pairs)
    r = np.sqrt(-2.0 * np.log(_uniform01(z[0::2])))
    th = 2.0 * math.pi * _uniform01(z[1::2])
    vals = np.empty(2 * pairs, dtype=np.float64)
    vals[0::2] = r * np.cos(th)
    vals[1::2] = r * np.sin(th)
    return vals[:n].astype(np.float32).astype(np.float16).view(np.uint16)


def scaled_normal_bf16(seed: int, tensor_id: int, n: int, std: float) -> np.ndarray:
    """N(0, std^2) samples rounded to bf16 bits (std applied in float32)."""
    v = bf16_bits_to_float32(normal_bf16(seed, tensor_id, n)) * np.float32(std)
    return float32_to_bf16_bits(v)


@dataclasses.dataclass
class PrologueInputs:
    base: DecodeInputs           # cache, block table and lengths (counting the new tokens)
    kv_new: np.ndarray           # uint16 [B, s_q, 576] rows of the new tokens
    q_nope: np.ndarray           # uint16 [B, s_q, h_q, 128]
    q_rope: np.ndarray           # uint16 [B, s_q, h_q, 64]
    w_uk: np.ndarray             # uint16 [h_q, 128, 512], N(0, 1/128)


def make_prologue_inputs(seed: int, batch: int, s_q: int, h_q: int, seqlens, *,
                         extra_pages: int = 0) -> PrologueInputs:
    base = make_inputs(seed, batch, s_q, h_q, seqlens, extra_pages=extra_pages, poison=False)
    kv_new = normal_bf16(seed, TENSOR_KV_NEW, batch * s_q * D_QK).reshape(batch, s_q, D_QK)
    q_nope = normal_bf16(seed, TENSOR_Q_NOPE, batch * s_q * h_q * D_NOPE).reshape(
        batch, s_q, h_q, D_NOPE)
    q_rope = normal_bf16(seed, TENSOR_Q_ROPE, batch * s_q * h_q * D_ROPE).reshape(
        batch, s_q, h_q, D_ROPE)
    w_uk = scaled_normal_bf16(seed, TENSOR_W_UK, h_q * D_NOPE * D_C, D_NOPE ** -0.5).reshape(
        h_q, D_NOPE, D_C)
    return PrologueInputs(base=base, kv_new=kv_new, q_nope=q_nope, q_rope=q_rope, w_uk=w_uk)


@dataclasses.dataclass
class PrologueWorkload:
    """Append + absorption at the shape of a decode workload."""
    name: str
    batch: int
    s_q: int
    h_q: int
    seqlen: int
    seed: int = 0

    def make(self) -> PrologueInputs:
        return make_prologue_inputs(self.seed, self.batch, self.s_q, self.h_q,
                                    np.full(self.batch, self.seqlen, dtype=np.int32))

    def absorb_flops(self) -> float:
        return 2.0 * self.batch * self.s_q * self.h_q * D_NOPE * D_C

    def absorb_bytes(self) -> float:
        """W_UK once, q_nope and q_rope read, the 576-wide query written."""
        rows = self.batch * self.s_q * self.h_q
        return float(self.h_q * D_NOPE * D_C * 2 + rows * (D_NOPE + D_ROPE) * 2 + rows * D_QK * 2)

    def append_bytes(self) -> float:
        """Each new row read once and written once."""
        return float(2 * self.batch * self.s_q * D_QK * 2)


PROLOGUE_WORKLOADS = {
    "prologue_b16_h128": PrologueWorkload("prologue_b16_h128", 16, 1, 128, 4096, seed=1),
    "prologue_b132_sq2_h128": PrologueWorkload("prologue_b132_sq2_h128", 132, 2, 128, 8192,
                                               seed=3),
}


@dataclasses.dataclass
class GemmWorkload:
    """C = A B with A [M, K], B [K, N] row-major, fp16 inputs N(0, 1)."""
    name: str
    M: int
    N: int
    K: int
    seed: int = 0

    def make(self):
        a = normal_f16(self.seed, TENSOR_GEMM_A, self.M * self.K).reshape(self.M, self.K)
        b = normal_f16(self.seed, TENSOR_GEMM_B, self.K * self.N).reshape(self.K, self.N)
        return a, b

    def flops(self) -> float:
        return 2.0 * self.M * self.N * self.K

    def bytes(self) -> float:
        return float(2 * (self.M * self.K + self.K * self.N + self.M * self.N))


# The GEMM tutorial's comparison: FP16, 2048 x 2048 x 2048.
GEMM_WORKLOADS = {"gemm_f16_2048": GemmWorkload("gemm_f16_2048", 2048, 2048, 2048, seed=6)}


# ---------------------------------------------------------------------------
# Dense attention forward (FlashAttention-style), [B, S, H, d] layouts.  The
# MLA prefill reading: DeepSeek's prefill runs attention in the MHA form,
# 128 heads with d_qk = 128 + 64 = 192 and d_v = 128, causal, scale 192^-0.5.
TENSOR_ATT_Q = 0x4151
TENSOR_ATT_K = 0x414B
TENSOR_ATT_V = 0x4156


@dataclasses.dataclass
class AttentionInputs:
    q: np.ndarray        # uint16 [B, S, H, d_qk]
    k: np.ndarray        # uint16 [B, S, H, d_qk]
    v: np.ndarray        # uint16 [B, S, H, d_v]
    causal: bool
    scale: float


def make_attention_inputs(seed: int, batch: int, seqlen: int, heads: int, d_qk: int, d_v: int,
                          causal: bool = True, scale: float | None = None) -> AttentionInputs:
    n_qk = batch * seqlen * heads * d_qk
    q = normal_bf16(seed, TENSOR_ATT_Q, n_qk).reshape(batch, seqlen, heads, d_qk)
    k = normal_bf16(seed, TENSOR_ATT_K, n_qk).reshape(batch, seqlen, heads, d_qk)
    v = normal_bf16(seed, TENSOR_ATT_V, batch * seqlen * heads * d_v).reshape(
        batch, seqlen, heads, d_v)
    return AttentionInputs(q=q, k=k, v=v, causal=causal,
                           scale=float(d_qk ** -0.5 if scale is None else scale))


@dataclasses.dataclass
class AttentionWorkload:
    name: str
    batch: int
    seqlen: int
    heads: int
    d_qk: int
    d_v: int
    causal: bool = True
    seed: int = 0

    def make(self) -> AttentionInputs:
        return make_attention_inputs(self.seed, self.batch, self.seqlen, self.heads, self.d_qk,
                                     self.d_v, self.causal)

    def pairs(self) -> float:
        """(query, key) pairs attended."""
        S = self.seqlen
        per = S * (S + 1) / 2 if self.causal else S * S
        return float(self.batch * self.heads * per)

    def flops(self) -> float:
        return 2.0 * (self.d_qk + self.d_v) * self.pairs()

    def bytes(self) -> float:
        rows = self.batch * self.seqlen * self.heads
        return float(rows * (2 * self.d_qk * 2 + self.d_v * 2 + self.d_v * 2 + 4))


ATTENTION_WORKLOADS = {
    # DeepSeek MLA prefill in the MHA form: one 4096-token sequence, 128 heads
    "prefill_b1_h128_s4096_d192": AttentionWorkload("prefill_b1_h128_s4096_d192", 1, 4096, 128,
                                                    192, 128, True, seed=8),
}
