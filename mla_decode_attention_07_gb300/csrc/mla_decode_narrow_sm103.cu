// MLA decode for few query rows per batch entry (s_q * h_q <= 32, e.g. the
// 16 or 32 heads per GPU of a model with 128 heads split over 8 or 4 GPUs,
// or two speculative tokens of 16 heads), sm_103a.
//
// What it computes is the paged MLA decode of mla_decode_sm103.cu (the same
// plan, the same partial results and combine, the same numerics): per query
// row, softmax(scale * q . k_t) over the visible cache rows k_t (576 dims),
// weighted sum of their first 512 dims, and lse.
//
// Why a second kernel.  The general kernel runs 128 query rows per tile on a
// CTA pair that exchanges partial scores and probabilities every page,
// because O for 128 rows x 512 dims fills a whole SM's TMEM.  With R <= 32
// rows the whole problem fits one SM:
//  * O is kept transposed: O^T = V^T P^T (M = 512 value dims in four blocks
//    of 128 TMEM lanes, N = R rows (16 or 32), K = 64 keys), 4 R TMEM
//    columns.  V^T is the page stage itself read as an M/N-major A operand;
//    P^T is an R x 64 K-major tile.
//  * S = Q K^T runs with M = 128: TMEM lane m holds query row m % R, so each
//    row appears in 128 / R lanes (Q is stored that many times in TMEM as the
//    A operand, 288 columns for 576 dims).  The tensor core does the extra
//    score work, which it has room for (the page is HBM-bound), and in
//    exchange the 128 softmax threads each read a different slice of a row
//    (64 R / 128 key columns) from TMEM in one load; the row max goes through
//    a small table of the four warps' maxima (one meeting per page).
//  * Each SM loads whole pages (72 KB, 9 boxes of 64 dims), three stages.
//    With R = 16 two score tiles fit in TMEM beside Q and O^T; with R = 32
//    one does (the next page's scores wait for this page's to be read).
// The plan gives each cluster (CTA pair) a page range, as for the general
// kernel; here the two CTAs take alternate pages of it and each runs its own
// online softmax.  At the end of an entry they merge: each writes the other's
// half of its O^T and its row statistics into rows of the split-partial
// workspace that a plan of at most R rows never uses (see rec_ptr), and
// signals the other through an mbarrier (release/acquire at cluster scope);
// each then finishes its half of the output dims.  The result (final output,
// or one partial per split) is exactly what the general kernel writes, so
// the combine is shared.
//
// Warp roles: warps 0-3 softmax, merge and epilogue (thread w * 32 + l owns
// TMEM lane w * 32 + l), warp 4 the TMA producer, warp 5 the score MMA issuer
// and TMEM owner, warp 6 the P.V MMA issuer.  Every wait is bounded
// (globaltimer): on expiry the kernel records MLA_ERR_DEVICE_TIMEOUT, tells
// the peer CTA, lets in-flight copies land, frees TMEM and returns.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <type_traits>

#include "mla.h"
#include "mla_internal.h"
#include "ptx_sm103.cuh"

namespace mla {
namespace {

constexpr int kNThreads = 224;
constexpr int kNSoftWarps = 4;
constexpr int kNSoftThreads = 32 * kNSoftWarps;
constexpr int kNProducerWarp = 4;
constexpr int kNMmaWarp = 5;      // score MMAs; owns TMEM
constexpr int kNPvWarp = 6;       // P.V MMAs
constexpr uint64_t kNWaitNs = 2000000000ull;  // 2 s per wait
constexpr uint64_t kNDrainNs = 2000000ull;    // settle time after an abort
constexpr float kNRescale = 8.0f;             // log2 units
constexpr float kNLn2 = 0.69314718055994530942f;

// Shared memory (offsets from a 1024-byte aligned base): three whole-page
// stages (72 KB each: nine 64-key x 64-dim boxes, 128-byte swizzle).
constexpr int kNStages = 3;
constexpr uint32_t kNBox = 8192;                        // 64 keys x 64 dims bf16, 128-byte swizzle
constexpr uint32_t kNBoxes = kDqk / 64;                 // 9
constexpr uint32_t kNStageBytes = kNBoxes * kNBox;      // one whole page
constexpr uint32_t kNTmemCols = 512;
constexpr uint32_t kNColQ = 0;                          // [0, 288): Q, bf16x2
constexpr uint32_t kNColS = 320;                        // score tiles, 64 columns each

// Everything that depends on the row count R (16 or 32).
template <int kR>
struct NShape {
  static_assert(kR == 16 || kR == 32, "16 or 32 query rows");
  static constexpr int kSlots = kNSoftThreads / kR;      // softmax threads per row (= kRep)
  static constexpr int kCols = 64 / kSlots;              // key columns per thread and page
  static constexpr int kSBufs = kR == 16 ? 2 : 1;        // score tiles in TMEM
  static constexpr uint32_t kColO = kR == 16 ? 448 : 384;   // O^T: 4 R columns
  static constexpr uint32_t kPBytes = (uint32_t)kR * 128u;  // P^T tile: R rows x 64 keys bf16
  static constexpr uint32_t kP = kNStages * kNStageBytes;   // 2 P^T tiles
  static constexpr uint32_t kPmax = kP + 2 * kPBytes;       // 2 x float[R][4 warps] page maxima
  static constexpr uint32_t kFlag = kPmax + 2 * (uint32_t)kR * 16u;   // u32: the peer has an O
  static constexpr uint32_t kBar = kFlag + 16;
  static constexpr uint32_t kMisc = kBar + 8 * 24;          // TMEM slot, abort flag
  static constexpr uint32_t kSmemAlloc = kMisc + 16 + 1024;
  // merge-time tables, in the P^T tiles (no P.V reads them then, and no
  // probabilities of the next entry are written before the merge ends)
  static constexpr uint32_t kSums = kP;                     // float[2][R][kSlots] l, lb
  static constexpr uint32_t kFac = kP + 1024;               // float[2][R] merge factors
  // merge records: rows [R, 128) of each 4-dim group of a partial slot
  static constexpr int kRecPerGroup = (kTileRows - kR) * 4 / kR;
  static_assert(kColO + 4 * kR <= kNTmemCols && kNColS + 64 * kSBufs <= kColO, "TMEM columns");
  static_assert(kP % 1024 == 0 && kPBytes % 1024 == 0, "swizzled buffers need 1 KB alignment");
  static_assert(2 * kPBytes >= 1024 + 8 * kR, "merge tables fit in the P^T tiles");
  static_assert(kSmemAlloc <= 232448, "shared memory");
  static_assert(259 / kRecPerGroup < kDv / 4, "merge records fit in the unused rows");
};

enum NBar : uint32_t {
  N_FULL = 0,                 // [3] page loaded (TMA tx)
  N_EMPTY = kNStages,         // [3] page consumed (MMA commit after its P.V)
  N_SFULL = 2 * kNStages,     // [2] score tile ready (MMA commit)
  N_SEMPTY = N_SFULL + 2,     // [2] score tile read (4 softmax warps)
  N_PFULL = N_SEMPTY + 2,     // [2] P^T written, O^T rescaled (4 softmax warps)
  N_PEMPTY = N_PFULL + 2,     // [2] the P.V of the tile's page done (MMA commit)
  N_QFULL = N_PEMPTY + 2,     // Q of the entry in TMEM (4 softmax warps)
  N_QEMPTY,                   // the entry's last score MMA done (MMA commit)
  N_MERGE,                    // the peer's records of the entry are written (remote arrive)
  N_MFREE,                    // the peer has read my records of the entry (remote arrive)
  N_SYNC,                     // the four softmax warps meet (one arrive per warp, every use)
  N_TEARDOWN,
  N_COUNT,
};
static_assert(N_COUNT <= 24, "barrier space");

// Merge records: sender rank r of cluster c writes into partial slot 2c + r,
// in the rows [R, 128) of each group of four dims, which a plan of at most R
// rows never uses.  Record k (R floats, one per row) sits in dim group
// k / kRecPerGroup after the group's first R rows.  Records 0-255: O^T of the
// receiver's 256 dims (relative dim order); 256-258: the sender's row max,
// sum of the fp32 probabilities and sum of the bf16 probabilities; 259: flag
// (float 1 if the sender had pages of the entry).
constexpr int kRecMax = 256, kRecL = 257, kRecLb = 258, kRecFlag = 259;
template <int kR>
__device__ __forceinline__ float* rec_ptr(float* ws_o, int cluster, uint32_t sender, int k) {
  constexpr int kPer = NShape<kR>::kRecPerGroup;
  return ws_o + (int64_t)(2 * cluster + (int)sender) * kSlotFloats +
         (int64_t)(k / kPer) * (kTileRows * 4) + 4 * kR + (k % kPer) * kR;
}

struct NCtx {
  uint32_t sbase, tmem, rank, peer, abort_addr, peer_abort_addr;
  uint32_t bar0;   // the first mbarrier
  int* err;
  __device__ __forceinline__ uint32_t bar(uint32_t i) const { return bar0 + 8u * i; }
};

__device__ __forceinline__ void n_abort(const NCtx& x) {
  atomicCAS(x.err, 0, MLA_ERR_DEVICE_TIMEOUT);
  ptx::st_shared_u32(x.abort_addr, 1u);
  ptx::st_cluster_u32(x.peer_abort_addr, 1u);
}

__device__ __forceinline__ bool n_wait(const NCtx& x, uint32_t bar, uint32_t parity,
                                       bool cluster_scope = false) {
  if (cluster_scope ? ptx::mbar_try_wait_cluster(bar, parity) : ptx::mbar_try_wait(bar, parity))
    return true;
  const uint64_t t0 = ptx::globaltimer();
  for (uint32_t i = 1;; ++i) {
    if (cluster_scope ? ptx::mbar_try_wait_cluster(bar, parity) : ptx::mbar_try_wait(bar, parity))
      return true;
    if ((i & 63u) == 0u) {
      if (ptx::ld_shared_u32_volatile(x.abort_addr) != 0u) return false;
      if (ptx::globaltimer() - t0 > kNWaitNs) {
        n_abort(x);
        return false;
      }
    }
  }
}
__device__ __forceinline__ bool n_wait_warp(const NCtx& x, uint32_t bar, uint32_t parity,
                                            bool cluster_scope = false) {
  const bool ok = n_wait(x, bar, parity, cluster_scope);
  return __all_sync(0xffffffffu, ok);
}

struct NWork {
  int b0, p0, b1, p1, split0, cluster;
  const int32_t* items;
};

// The four softmax warps meet: a barrier whose wait is bounded (a warp that
// gave up does not leave the others waiting).  Shared-memory writes before
// it are visible after it.  `uses` counts the meetings so far.
__device__ __forceinline__ bool n_sync(const NCtx& x, uint32_t& uses, int lane) {
  __syncwarp();
  if (lane == 0) ptx::mbar_arrive(x.bar(N_SYNC));
  const bool ok = n_wait_warp(x, x.bar(N_SYNC), uses & 1u);
  ++uses;
  return ok;
}

// Pages of segment [pb, pe) taken by CTA `rank`: pb + rank, pb + rank + 2, ...
__device__ __forceinline__ int own_pages(int pb, int pe, uint32_t rank) {
  const int n = pe - pb - (int)rank;
  return n > 0 ? (n + 1) / 2 : 0;
}

// ------------------------------------------------------------------ producer
// This CTA's pages of the cluster's range, in order (g counts them), with
// the boundaries of their entries.
struct OwnPages {
  SegIter it;
  uint32_t rank, g;
  int b, pb, k, n_own;
  bool valid;
  __device__ __forceinline__ void init(const NWork& w, uint32_t r) {
    it = SegIter{w.b0, w.p0, w.b1, w.p1, w.items};
    rank = r;
    g = 0;
    next_entry();
  }
  __device__ __forceinline__ void next_entry() {
    int pe;
    valid = false;
    while (it.next(b, pb, pe)) {
      n_own = own_pages(pb, pe, rank);
      if (n_own > 0) {
        k = 0;
        valid = true;
        return;
      }
    }
  }
  __device__ __forceinline__ void advance() {
    ++g;
    if (++k == n_own) next_entry();
  }
  // the cursor's page within its entry
  __device__ __forceinline__ int page_index() const { return pb + (int)rank + 2 * k; }
};

__device__ __forceinline__ int n_page_of(const DecodeParams& prm, int b, int pg) {
  return pg < prm.max_pages ? prm.block_table[(size_t)b * prm.max_pages + pg] : -1;
}

__device__ __forceinline__ bool n_producer(const NCtx& x, const NWork& w, const DecodeParams& prm,
                                           const CUtensorMap* tm_kv) {
  const uint64_t policy = ptx::policy_evict_first();
  OwnPages cur;
  cur.init(w, x.rank);
  while (cur.valid) {
    // Entries past max_pages are never read: such a page is reported and
    // served from page 0.
    int page = n_page_of(prm, cur.b, cur.page_index());
    const uint32_t g = cur.g, s = g % kNStages;
    if (!n_wait(x, x.bar(N_EMPTY + s), ((g / kNStages) & 1u) ^ 1u)) return false;
    if ((unsigned)page >= (unsigned)prm.num_pages) {
      atomicCAS(x.err, 0, MLA_ERR_DEVICE_BOUNDS);
      page = 0;
    }
    ptx::mbar_arrive_expect_tx(x.bar(N_FULL + s), kNStageBytes);
    const uint32_t st = x.sbase + s * kNStageBytes;
#pragma unroll 1
    for (uint32_t j = 0; j < kNBoxes; ++j)
      ptx::tma_load_2d_hint(st + j * kNBox, tm_kv, 64 * (int32_t)j, page * kPageTokens,
                            x.bar(N_FULL + s), policy);
    cur.advance();
  }
  return true;
}

// ------------------------------------------------------------------ MMA issuer
// Two issuing warps feed the tensor pipe: issuing a page's 36 score MMAs
// blocks a warp for most of their run time (the MMA queue pushes back), so a
// single issuer would hold a finished page's P.V (and with it the page's
// stage) behind the next page's scores.  Each warp commits its own MMAs.
//
// Score issuer: S(g) = Q K^T once page g is loaded, its score tile is free
// and the entry's Q is in TMEM.
template <int kR>
__device__ __forceinline__ bool n_mma_s(const NCtx& x, const NWork& w) {
  using S = NShape<kR>;
  constexpr uint32_t id_s = ptx::idesc_bf16_f32(128, 64, 0, 0);
  OwnPages sc;
  sc.init(w, x.rank);
  uint32_t sq = 0;   // entries whose score MMAs are all issued (Q uses)
  while (sc.valid) {
    const uint32_t g = sc.g, s = g % kNStages;
    if (sc.k == 0 && !n_wait_warp(x, x.bar(N_QFULL), sq & 1u)) return false;
    if (!n_wait_warp(x, x.bar(N_FULL + s), (g / kNStages) & 1u)) return false;
    // the score tile is free once the softmax has read the page that used it
    const uint32_t sb = g % S::kSBufs, su = g / S::kSBufs;
    if (su >= 1 && !n_wait_warp(x, x.bar(N_SEMPTY + sb), (su & 1u) ^ 1u)) return false;
    ptx::tc_fence_after();
    const uint32_t st = x.sbase + s * kNStageBytes;
    const uint32_t d_s = x.tmem + kNColS + sb * 64u;
#pragma unroll
    for (uint32_t kk = 0; kk < 4 * kNBoxes; ++kk) {
      const uint64_t bd =
          ptx::smem_desc(st + (kk >> 2) * kNBox + (kk & 3u) * 32u, 16, 1024, ptx::kLayoutSw128);
      ptx::mma_ts_elect(d_s, x.tmem + kNColQ + 8u * kk, bd, id_s, kk ? 1u : 0u);
    }
    ptx::mma_commit_elect(x.bar(N_SFULL + sb));
    if (sc.k == sc.n_own - 1) {
      ptx::mma_commit_elect(x.bar(N_QEMPTY));
      ++sq;
    }
    sc.advance();
  }
  return true;
}

// P.V issuer: O^T += V^T P^T once page g's probabilities are written; its
// commit hands the stage back to the producer and the P^T buffer to the
// softmax warps.
template <int kR>
__device__ __forceinline__ bool n_mma_o(const NCtx& x, const NWork& w) {
  using S = NShape<kR>;
  constexpr uint32_t id_o = ptx::idesc_bf16_f32(128, kR, 1, 0);   // A = V^T, M/N-major
  OwnPages oc;
  oc.init(w, x.rank);
  while (oc.valid) {
    const uint32_t gp = oc.g;
    if (!n_wait_warp(x, x.bar(N_PFULL + (gp & 1u)), (gp >> 1) & 1u)) return false;
    ptx::tc_fence_after();
    const bool first = (oc.k == 0);
    const uint32_t st = x.sbase + (gp % kNStages) * kNStageBytes;
    const uint32_t pt = x.sbase + S::kP + (gp & 1u) * S::kPBytes;
#pragma unroll
    for (uint32_t mb = 0; mb < 4; ++mb) {
#pragma unroll
      for (uint32_t k = 0; k < 4; ++k) {
        // V^T block mb: value dims [128 mb, +128) = boxes 2 mb, 2 mb + 1 (8 KB
        // apart along M), keys [16 k, +16): two 8-key groups 1 KB apart
        const uint64_t ad =
            ptx::smem_desc(st + 2u * mb * kNBox + k * 2048u, kNBox, 1024, ptx::kLayoutSw128);
        // P^T: R rows of 64 keys (128 bytes), 8-row groups 1 KB apart
        const uint64_t bd = ptx::smem_desc(pt + k * 32u, 16, 1024, ptx::kLayoutSw128);
        ptx::mma_ss_elect(x.tmem + S::kColO + (uint32_t)kR * mb, ad, bd, id_o,
                          (first && k == 0) ? 0u : 1u);
      }
    }
    ptx::mma_commit_elect(x.bar(N_EMPTY + gp % kNStages));
    ptx::mma_commit_elect(x.bar(N_PEMPTY + (gp & 1u)));
    oc.advance();
  }
  return true;
}

// ------------------------------------------------------------------ softmax
// Thread (warp q, lane l), TMEM lane t = 32 q + l: query row i = l % R, slot
// t / R of the row's 128 / R threads, key columns [slot * cols, +cols) of
// every page (cols = 64 R / 128); in the merge and epilogue, value dims
// 128 j + t.
template <int kR>
__device__ __forceinline__ bool n_softmax(const NCtx& x, const NWork& w, const DecodeParams& prm,
                                          int warp, int lane) {
  using S = NShape<kR>;
  constexpr int kC = S::kCols;
  const int tl = 32 * warp + lane;                        // TMEM lane
  const int i = lane % kR;                                // query row
  const int slot = tl / kR;
  const int col0 = slot * kC;                             // this thread's key columns
  const uint32_t lanes = (uint32_t)(32 * warp) << 16;
  const int R = prm.s_q * prm.h_q;
  const bool valid = i < R;
  const int qi = valid ? i / prm.h_q : 0;
  const float sl2 = prm.scale_log2;
  const __nv_bfloat16* q = static_cast<const __nv_bfloat16*>(prm.q);
  // P^T row i, 16-byte chunks col0 / 8 .. (128-byte swizzle)
  const uint32_t prow = (uint32_t)i * 128u;
  const uint32_t pswz = (uint32_t)i & 7u;
  const uint32_t peer_merge = ptx::map_to_rank(x.bar(N_MERGE), x.peer);
  const uint32_t peer_mfree = ptx::map_to_rank(x.bar(N_MFREE), x.peer);

  SegIter it{w.b0, w.p0, w.b1, w.p1, w.items};
  int b, pb, pe;
  uint32_t g = 0, nq = 0, n_item = 0, uses = 0;
  // Q row i of entry qb into this lane's 288 columns, once the previous
  // entry's last score MMA is done (two rounds of 40 and 32 loads in
  // flight).  The next entry's Q is loaded before this entry's merge, so its
  // first score MMA runs while the merge does.
  auto load_q = [&](int qb) -> bool {
    if (!n_wait_warp(x, x.bar(N_QEMPTY), (nq & 1u) ^ 1u)) return false;
    const uint4* src = reinterpret_cast<const uint4*>(q + ((int64_t)qb * R + (valid ? i : 0)) * kDqk);
    // 72 pieces of 16 bytes = 9 chunks of 32 columns: chunks 0-4, then 5-8
    auto round = [&](auto c0_tag, auto nc_tag) {
      constexpr int c0 = decltype(c0_tag)::value, nc = decltype(nc_tag)::value;
      uint4 qv[8 * nc];
#pragma unroll
      for (int j = 0; j < 8 * nc; ++j) qv[j] = valid ? src[8 * c0 + j] : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
      for (int ch = 0; ch < nc; ++ch) {
        uint32_t v[32];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          v[4 * j] = qv[8 * ch + j].x;
          v[4 * j + 1] = qv[8 * ch + j].y;
          v[4 * j + 2] = qv[8 * ch + j].z;
          v[4 * j + 3] = qv[8 * ch + j].w;
        }
        ptx::tmem_st32(x.tmem + lanes + kNColQ + (uint32_t)(c0 + ch) * 32u, v);
      }
    };
    round(std::integral_constant<int, 0>{}, std::integral_constant<int, 5>{});
    round(std::integral_constant<int, 5>{}, std::integral_constant<int, 4>{});
    ptx::tmem_wait_st();
    ptx::tc_fence_before();
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive(x.bar(N_QFULL));
    ++nq;
    return true;
  };
  bool have = it.next(b, pb, pe);
  if (have && own_pages(pb, pe, x.rank) > 0 && !load_q(b)) return false;
  while (have) {
    const int n_own = own_pages(pb, pe, x.rank);
    const int L = prm.seqlens[b];
    const int n_valid = valid ? L - prm.s_q + 1 + qi : 0;   // keys visible to row i
    const int P_total = w.items[b * kItemWords + 0];
    float m_ref = -INFINITY, l_run = 0.f, lb_run = 0.f;   // row i's reference max and sums

    for (int k = 0; k < n_own; ++k, ++g) {
      const int pg = pb + (int)x.rank + 2 * k;
      const uint32_t pbf = g & 1u;                          // P^T tile and page-max table
      const uint32_t sb = g % S::kSBufs, su = g / S::kSBufs;   // score tile and its use
      if (!n_wait_warp(x, x.bar(N_SFULL + sb), su & 1u)) return false;
      ptx::tc_fence_after();
      float mine[kC];
      if constexpr (kR == 16) {
        // lanes 32 q + [0, 16) (rows 0-15): columns 16 q + [0, 8) to the
        // first half-warp, 16 q + [8, 16) to the second
        uint32_t v8[8];
        ptx::tmem_ld16x2_x8_wait<8>(x.tmem + lanes + kNColS + sb * 64u + 16u * (uint32_t)warp, v8);
#pragma unroll
        for (int j = 0; j < 8; ++j) mine[j] = __uint_as_float(v8[j]);
      } else {
        // this lane (row l), columns 16 q + [0, 16)
        uint32_t v16[16];
        ptx::tmem_ld32x16_wait(x.tmem + lanes + kNColS + sb * 64u + 16u * (uint32_t)warp, v16);
#pragma unroll
        for (int j = 0; j < 16; ++j) mine[j] = __uint_as_float(v16[j]);
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(x.bar(N_SEMPTY + sb));
      // keys past the row's visible count get no weight
      const int t0 = pg * kPageTokens + col0;
#pragma unroll
      for (int j = 0; j < kC; ++j)
        if (t0 + j >= n_valid) mine[j] = -INFINITY;
      // Row max of the page: this thread's columns (and, for R = 16, its
      // half-warp partner's), then the four warps' maxima through shared
      // memory (double buffered by page parity, one meeting per page).
      float pm = mine[0];
#pragma unroll
      for (int j = 1; j < kC; ++j) pm = fmaxf(pm, mine[j]);
      if constexpr (kR == 16) pm = fmaxf(pm, __shfl_xor_sync(0xffffffffu, pm, 16));
      const uint32_t pmax = x.sbase + S::kPmax + pbf * (uint32_t)kR * 16u;   // float[R][4 warps]
      if (lane < kR) ptx::st_shared_u32(pmax + (uint32_t)(i * 4 + warp) * 4u, __float_as_uint(pm));
      if (!n_sync(x, uses, lane)) return false;
      // Lazy rescale (log2 domain): the reference max of a row moves only when
      // its max grows by more than 2^8.  Each thread decides for its own row
      // (all threads of a row read the same four numbers); every warp holds
      // every row, so a rescale of any row is seen warp-wide.
      float a_own = 1.0f;
      bool resc = false;
      {
        const uint4 p4 = ptx::ld_shared_v4u(pmax + (uint32_t)i * 16u);
        const float mx = fmaxf(fmaxf(__uint_as_float(p4.x), __uint_as_float(p4.y)),
                               fmaxf(__uint_as_float(p4.z), __uint_as_float(p4.w)));
        const float m_cand = fmaxf(m_ref, mx * sl2);   // sl2 > 0
        if (k == 0) {
          m_ref = m_cand;
        } else if (m_cand > m_ref + kNRescale) {
          a_own = ptx::ex2(m_ref - m_cand);
          m_ref = m_cand;
          resc = true;
        }
      }
      const bool any = __any_sync(0xffffffffu, resc);
      l_run *= a_own;
      lb_run *= a_own;
      const float neg_m = (m_ref == -INFINITY) ? 0.f : -m_ref;
      uint32_t pk[kC / 2];
#pragma unroll
      for (int j = 0; j < kC / 2; ++j) {
        const float a = ptx::ex2(fmaf(mine[2 * j], sl2, neg_m));
        const float c = ptx::ex2(fmaf(mine[2 * j + 1], sl2, neg_m));
        pk[j] = ptx::pack_bf16x2(a, c);
        l_run += a + c;
        lb_run += __uint_as_float(pk[j] << 16) + __uint_as_float(pk[j] & 0xffff0000u);
      }
      // P^T buffer g % 2 is free once the P.V of page g - 2 is done
      if (g >= 2 && !n_wait_warp(x, x.bar(N_PEMPTY + pbf), ((g >> 1) & 1u) ^ 1u)) return false;
      // Past the end of the sequence the last page's slots hold stale data:
      // their probabilities are 0, but 0 * NaN is NaN in the P.V MMA, so
      // zero those value rows first (latent boxes 0-7 of the stage).
      if (pg == P_total - 1 && (L & (kPageTokens - 1)) != 0) {
        const int tz = L & (kPageTokens - 1);
        const uint32_t st = x.sbase + (g % kNStages) * kNStageBytes;
        const int n16 = (kPageTokens - tz) * 8 * 8;   // rows x 8 boxes x 8 pieces of 16 bytes
        for (int idx = tl; idx < n16; idx += kNSoftThreads) {
          const int row = tz + (idx >> 6), box = (idx >> 3) & 7, c16 = idx & 7;
          ptx::st_shared_v4(st + box * kNBox + row * 128 + c16 * 16, 0u, 0u, 0u, 0u);
        }
      }
      {
        const uint32_t pt = x.sbase + S::kP + pbf * S::kPBytes + prow;
#pragma unroll
        for (int c = 0; c < kC / 8; ++c) {
          const uint32_t chunk = (uint32_t)(col0 / 8 + c);
          ptx::st_shared_v4(pt + ((chunk ^ pswz) << 4), pk[4 * c], pk[4 * c + 1], pk[4 * c + 2],
                            pk[4 * c + 3]);
        }
      }
      ptx::fence_proxy_async_smem();
      // O^T column r (of each 128-dim block) holds row r: rescale the columns
      // whose factor is not 1 (after the P.V of page g - 1 is done; this
      // page's P.V waits for us)
      if (any) {
        float al[kR];   // row r's factor, from lane r
#pragma unroll
        for (int r = 0; r < kR; ++r) al[r] = __shfl_sync(0xffffffffu, a_own, r);
        if (!n_wait_warp(x, x.bar(N_PEMPTY + (pbf ^ 1u)), ((g - 1) >> 1) & 1u)) return false;
        ptx::tc_fence_after();
#pragma unroll 1
        for (int h2 = 0; h2 < 4 * kR / 32; ++h2) {
          uint32_t o[32];
          ptx::tmem_ld32_wait(x.tmem + lanes + S::kColO + 32u * (uint32_t)h2, o);
#pragma unroll
          for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * al[j % kR]);
          ptx::tmem_st32(x.tmem + lanes + S::kColO + 32u * (uint32_t)h2, o);
        }
        ptx::tmem_wait_st();
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(x.bar(N_PFULL + pbf));
    }
    // the next entry's Q (its first score MMA then overlaps this merge)
    int nb = 0, npb = 0, npe = 0;
    const bool nhave = it.next(nb, npb, npe);
    if (nhave && own_pages(npb, npe, x.rank) > 0 && !load_q(nb)) return false;

    // ---- merge with the peer, then this CTA's half of the output dims ----
    const bool has = n_own > 0;
    // O^T blocks 2 rank, 2 rank + 1 (this CTA's output dims) and the peer's two
    float own[2 * kR], oth[2 * kR];
    if (has) {
      // every P.V of the entry is done once the last page's is
      const uint32_t gl = g - 1;
      if (!n_wait_warp(x, x.bar(N_PEMPTY + (gl & 1u)), (gl >> 1) & 1u)) return false;
      ptx::tc_fence_after();
#pragma unroll
      for (int h2 = 0; h2 < 2 * kR / 32; ++h2) {
        uint32_t v[32];
        ptx::tmem_ld32_wait(x.tmem + lanes + S::kColO + 2u * kR * x.rank + 32u * h2, v);
#pragma unroll
        for (int j = 0; j < 32; ++j) own[32 * h2 + j] = __uint_as_float(v[j]);
        ptx::tmem_ld32_wait(x.tmem + lanes + S::kColO + 2u * kR * x.peer + 32u * h2, v);
#pragma unroll
        for (int j = 0; j < 32; ++j) oth[32 * h2 + j] = __uint_as_float(v[j]);
      }
    } else {
#pragma unroll
      for (int j = 0; j < 2 * kR; ++j) own[j] = oth[j] = 0.f;
    }
    // the peer has read the records of my previous entry
    if (n_item > 0 && !n_wait_warp(x, x.bar(N_MFREE), (n_item - 1) & 1u, true)) return false;
    if (has) {
      // the peer's dims: blocks 2 peer, 2 peer + 1 -> records 0-255 (relative)
#pragma unroll
      for (int jb = 0; jb < 2; ++jb) {
        float4* rec = reinterpret_cast<float4*>(rec_ptr<kR>(prm.ws_o, w.cluster, x.rank, 128 * jb + tl));
#pragma unroll
        for (int r4 = 0; r4 < kR / 4; ++r4)
          rec[r4] = make_float4(oth[kR * jb + 4 * r4], oth[kR * jb + 4 * r4 + 1],
                                oth[kR * jb + 4 * r4 + 2], oth[kR * jb + 4 * r4 + 3]);
      }
    }
    // the row sums over the row's threads (in the P^T tiles, idle now)
    ptx::st_shared_u32(x.sbase + S::kSums + (uint32_t)(i * S::kSlots + slot) * 4u, __float_as_uint(l_run));
    ptx::st_shared_u32(x.sbase + S::kSums + 512u + (uint32_t)(i * S::kSlots + slot) * 4u,
                       __float_as_uint(lb_run));
    if (!n_sync(x, uses, lane)) return false;
    float l_tot = 0.f, lb_tot = 0.f;
    if (tl < kR) {   // warp 0, lane = row
#pragma unroll
      for (int j = 0; j < S::kSlots; ++j) {
        l_tot += __uint_as_float(ptx::ld_shared_u32_volatile(x.sbase + S::kSums + (uint32_t)(i * S::kSlots + j) * 4u));
        lb_tot += __uint_as_float(ptx::ld_shared_u32_volatile(x.sbase + S::kSums + 512u + (uint32_t)(i * S::kSlots + j) * 4u));
      }
      rec_ptr<kR>(prm.ws_o, w.cluster, x.rank, kRecMax)[i] = has ? m_ref : -INFINITY;
      rec_ptr<kR>(prm.ws_o, w.cluster, x.rank, kRecL)[i] = l_tot;
      rec_ptr<kR>(prm.ws_o, w.cluster, x.rank, kRecLb)[i] = lb_tot;
      if (i == 0) rec_ptr<kR>(prm.ws_o, w.cluster, x.rank, kRecFlag)[0] = has ? 1.0f : 0.0f;
    }
    __threadfence();
    if (!n_sync(x, uses, lane)) return false;
    if (warp == 0 && lane == 0) ptx::mbar_arrive_cluster_release(peer_merge);
    if (!n_wait_warp(x, x.bar(N_MERGE), n_item & 1u, true)) return false;

    // Row factors: both halves scaled to the common max, with 1/l.  The row
    // threads of warp 0 also write lse.
    const int ns = w.items[b * kItemWords + 1];
    const bool direct = (ns == 1);
    const int sidx = (n_item == 0) ? w.split0 : 0;
    const int64_t slot_o = (int64_t)w.items[b * kItemWords + 2] + sidx;   // one tile
    if (tl < kR) {
      const float m_p = __ldcg(rec_ptr<kR>(prm.ws_o, w.cluster, x.peer, kRecMax) + i);
      const float l_p = __ldcg(rec_ptr<kR>(prm.ws_o, w.cluster, x.peer, kRecL) + i);
      const float lb_p = __ldcg(rec_ptr<kR>(prm.ws_o, w.cluster, x.peer, kRecLb) + i);
      const float m_o = has ? m_ref : -INFINITY;
      const float m = fmaxf(m_o, m_p);
      const float fo = (m_o == -INFINITY) ? 0.f : ptx::ex2(m_o - m);
      const float fp = (m_p == -INFINITY) ? 0.f : ptx::ex2(m_p - m);
      const float lt = l_tot * fo + l_p * fp;
      const float lbt = lb_tot * fo + lb_p * fp;
      const float inv = lbt > 0.f ? 1.0f / lbt : 0.f;
      ptx::st_shared_u32(x.sbase + S::kFac + 4u * (uint32_t)i, __float_as_uint(fo * inv));
      ptx::st_shared_u32(x.sbase + S::kFac + 4u * kR + 4u * (uint32_t)i, __float_as_uint(fp * inv));
      if (i == 0)
        ptx::st_shared_u32(x.sbase + S::kFlag,
                           __ldcg(rec_ptr<kR>(prm.ws_o, w.cluster, x.peer, kRecFlag)) != 0.f ? 1u : 0u);
      if (x.rank == 0 && valid) {
        const float lse_v = lt > 0.f ? (m + log2f(lt)) * kNLn2 : -INFINITY;
        const int hh = i - qi * prm.h_q;
        if (direct)
          prm.lse[((int64_t)b * prm.h_q + hh) * prm.s_q + qi] = lse_v;
        else
          prm.ws_lse[slot_o * kTileRows + i] = lse_v;
      }
    }
    if (!n_sync(x, uses, lane)) return false;
    float fo[kR], fp[kR];
#pragma unroll
    for (int j = 0; j < kR / 4; ++j) {
      const uint4 a = ptx::ld_shared_v4u(x.sbase + S::kFac + 16u * (uint32_t)j);
      const uint4 c = ptx::ld_shared_v4u(x.sbase + S::kFac + 4u * kR + 16u * (uint32_t)j);
      fo[4 * j] = __uint_as_float(a.x);
      fo[4 * j + 1] = __uint_as_float(a.y);
      fo[4 * j + 2] = __uint_as_float(a.z);
      fo[4 * j + 3] = __uint_as_float(a.w);
      fp[4 * j] = __uint_as_float(c.x);
      fp[4 * j + 1] = __uint_as_float(c.y);
      fp[4 * j + 2] = __uint_as_float(c.z);
      fp[4 * j + 3] = __uint_as_float(c.w);
    }
    const bool peer_has = ptx::ld_shared_u32_volatile(x.sbase + S::kFlag) != 0u;
#pragma unroll
    for (int jb = 0; jb < 2; ++jb) {
      const int mb = 2 * (int)x.rank + jb;
      float op[kR];
      if (peer_has) {
        const float4* rec =
            reinterpret_cast<const float4*>(rec_ptr<kR>(prm.ws_o, w.cluster, x.peer, 128 * jb + tl));
#pragma unroll
        for (int r4 = 0; r4 < kR / 4; ++r4) {
          const float4 v4 = __ldcg(rec + r4);
          op[4 * r4] = v4.x;
          op[4 * r4 + 1] = v4.y;
          op[4 * r4 + 2] = v4.z;
          op[4 * r4 + 3] = v4.w;
        }
      } else {
#pragma unroll
        for (int j = 0; j < kR; ++j) op[j] = 0.f;
      }
      const int d = 128 * mb + tl;
#pragma unroll
      for (int r = 0; r < kR; ++r) {
        if (r >= R) break;
        const float val = own[kR * jb + r] * fo[r] + op[r] * fp[r];
        if (direct) {
          const int64_t oi = ((int64_t)b * R + r) * kDv + d;
          if (prm.out_f32)
            static_cast<float*>(prm.out)[oi] = val;
          else
            static_cast<__nv_bfloat16*>(prm.out)[oi] = __float2bfloat16_rn(val);
        } else {
          prm.ws_o[slot_o * kSlotFloats + (int64_t)(d >> 2) * (kTileRows * 4) + r * 4 + (d & 3)] = val;
        }
      }
    }
    // my reads of the peer's records (and of the tables in the P^T tiles)
    // are done
    if (!n_sync(x, uses, lane)) return false;
    if (warp == 0 && lane == 0) ptx::mbar_arrive_cluster_release(peer_mfree);
    ++n_item;
    b = nb;
    pb = npb;
    pe = npe;
    have = nhave;
  }
  return true;
}

template <int kR>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kNThreads, 1)
    mla_decode_narrow_kernel(const __grid_constant__ CUtensorMap tm_kv, const DecodeParams prm) {
  using S = NShape<kR>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  NCtx x;
  x.sbase = (ptx::smem_addr(smem_raw) + 1023u) & ~1023u;
  x.rank = ptx::cluster_ctarank();
  x.peer = x.rank ^ 1u;
  x.bar0 = x.sbase + S::kBar;
  x.abort_addr = x.sbase + S::kMisc + 4;
  x.peer_abort_addr = ptx::map_to_rank(x.abort_addr, x.peer);
  x.err = prm.err;
  const uint32_t tmem_slot = x.sbase + S::kMisc;
  const int cluster = (int)(blockIdx.x >> 1);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kNStages; ++s) {
      ptx::mbar_init(x.bar(N_FULL + s), 1);
      ptx::mbar_init(x.bar(N_EMPTY + s), 1);
    }
    for (int s = 0; s < 2; ++s) {
      ptx::mbar_init(x.bar(N_SFULL + s), 1);
      ptx::mbar_init(x.bar(N_SEMPTY + s), kNSoftWarps);
      ptx::mbar_init(x.bar(N_PFULL + s), kNSoftWarps);
      ptx::mbar_init(x.bar(N_PEMPTY + s), 1);
    }
    ptx::mbar_init(x.bar(N_QFULL), kNSoftWarps);
    ptx::mbar_init(x.bar(N_QEMPTY), 1);
    ptx::mbar_init(x.bar(N_MERGE), 1);
    ptx::mbar_init(x.bar(N_MFREE), 1);
    ptx::mbar_init(x.bar(N_SYNC), kNSoftWarps);
    ptx::mbar_init(x.bar(N_TEARDOWN), 2);   // both issuing warps
    ptx::st_shared_u32(x.abort_addr, 0u);
    ptx::fence_mbarrier_init();
  }
  if (warp == kNMmaWarp) {
    ptx::tmem_alloc(tmem_slot, kNTmemCols);
    ptx::tmem_relinquish();
  }
  if (warp == kNProducerWarp && lane == 0) ptx::prefetch_tmap(&tm_kv);
  ptx::tc_fence_before();
  ptx::cluster_sync();   // both CTAs' barriers initialised and TMEM allocated
  ptx::tc_fence_after();
  x.tmem = ptx::ld_shared_u32_volatile(tmem_slot);

  // The plan (and the inputs) come from earlier kernels on the stream.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  // The plan must describe this call (one tile: at most R query rows).
  const int32_t* plan = prm.plan;
  NWork w = {};
  bool has_work = false;
  const int nclusters = (int)(gridDim.x >> 1);
  const int gt_l = plan_group_clusters(nclusters, 1);
  const int32_t* cl = plan + H_WORDS + cluster * kClusterWords;
  const int e_b0 = cl[0], e_p0 = cl[1], e_b1 = cl[2], e_p1 = cl[3], e_s0 = cl[4];
  if (plan[H_MAGIC] != kPlanMagic || plan[H_BATCH] != prm.batch || plan[H_SQ] != prm.s_q ||
      plan[H_HQ] != prm.h_q || plan[H_NCLUSTERS] != nclusters || plan[H_GT] != gt_l ||
      plan[H_TILES] != 1 || gt_l <= 0 || prm.s_q * prm.h_q > kR) {
    if (threadIdx.x == 0 && x.rank == 0) atomicCAS(prm.err, 0, MLA_ERR_PLAN);
  } else if (cluster < plan[H_GUSED]) {
    w.b0 = e_b0;
    w.p0 = e_p0;
    w.b1 = e_b1;
    w.p1 = e_p1;
    w.split0 = e_s0;
    w.cluster = cluster;
    if (w.b0 < 0 || w.p0 < 0 || w.p1 < 0 || w.b0 > w.b1 || w.b1 > prm.batch ||
        (w.b1 == prm.batch && w.p1 != 0)) {
      if (threadIdx.x == 0 && x.rank == 0) atomicCAS(prm.err, 0, MLA_ERR_PLAN);
    } else if (!(w.b0 == w.b1 && w.p0 >= w.p1)) {
      has_work = true;
      w.items = plan + plan_off_items(gt_l) / 4;
    }
  }

  if (!has_work) {
    // nothing to do: fall through to the teardown
  } else if (warp == kNProducerWarp) {
    if (lane == 0) n_producer(x, w, prm, &tm_kv);
    __syncwarp();
  } else if (warp == kNMmaWarp) {
    n_mma_s<kR>(x, w);   // whole warp: one elected lane issues
    __syncwarp();
  } else if (warp == kNPvWarp) {
    n_mma_o<kR>(x, w);
    __syncwarp();
  } else {
    n_softmax<kR>(x, w, prm, warp, lane);
    __syncwarp();
  }

  // Teardown.  After an abort, give in-flight copies and MMAs time to land
  // before the shared memory and TMEM are released.
  const bool aborted = ptx::ld_shared_u32_volatile(x.abort_addr) != 0u;
  if (warp == kNMmaWarp || warp == kNPvWarp) {
    // each issuing warp's MMAs are done
    ptx::mma_commit_elect(x.bar(N_TEARDOWN));
    const uint64_t t0 = ptx::globaltimer();
    while (!ptx::mbar_try_wait(x.bar(N_TEARDOWN), 0u)) {
      if (ptx::globaltimer() - t0 > kNWaitNs) {
        if (lane == 0) atomicCAS(x.err, 0, MLA_ERR_DEVICE_TIMEOUT);
        break;
      }
    }
  }
  if (aborted) {
    const uint64_t t0 = ptx::globaltimer();
    while (ptx::globaltimer() - t0 < kNDrainNs) __nanosleep(1000);
  }
  __syncwarp();
  ptx::tc_fence_before();
  ptx::cluster_sync();   // no remote traffic into either CTA after this point
  if (warp == kNMmaWarp) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(x.tmem, kNTmemCols);
  }
}

}  // namespace

// At most 32 query rows, and enough pages for the CTA pair's per-entry merge
// (about 3 us: the partial O^T through L2 and a handshake) to pay off: the
// pair runs a cluster's pages about 1.7x faster than the general kernel, so
// calls whose block table holds at most 4 pages per cluster (latency-bound
// either way) stay on the general kernel.
bool narrow_decode_shape(int s_q, int h_q, int batch, int max_pages, int num_clusters) {
  return s_q * h_q <= 32 && (int64_t)batch * max_pages > 4 * (int64_t)num_clusters;
}

cudaError_t narrow_kernel_setup() {
  const cudaError_t e =
      cudaFuncSetAttribute(mla_decode_narrow_kernel<16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)NShape<16>::kSmemAlloc);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(mla_decode_narrow_kernel<32>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)NShape<32>::kSmemAlloc);
}

int narrow_max_clusters() {
  int n = -1;
  for (int k = 0; k < 2; ++k) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * 1024, 1, 1);
    cfg.blockDim = dim3(kNThreads, 1, 1);
    cfg.dynamicSmemBytes = k == 0 ? (size_t)NShape<16>::kSmemAlloc : (size_t)NShape<32>::kSmemAlloc;
    int m = 0;
    const cudaError_t e = k == 0 ? cudaOccupancyMaxActiveClusters(&m, mla_decode_narrow_kernel<16>, &cfg)
                                 : cudaOccupancyMaxActiveClusters(&m, mla_decode_narrow_kernel<32>, &cfg);
    if (e != cudaSuccess) return -1;
    n = (n < 0 || m < n) ? m : n;
  }
  return n;
}

cudaError_t launch_decode_narrow(const CUtensorMap& kv_map, const DecodeParams& p, int num_clusters,
                                 cudaStream_t stream) {
  const bool r16 = p.s_q * p.h_q <= 16;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * num_clusters);
  cfg.blockDim = dim3(kNThreads);
  cfg.dynamicSmemBytes = r16 ? NShape<16>::kSmemAlloc : NShape<32>::kSmemAlloc;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return r16 ? cudaLaunchKernelEx(&cfg, mla_decode_narrow_kernel<16>, kv_map, p)
             : cudaLaunchKernelEx(&cfg, mla_decode_narrow_kernel<32>, kv_map, p);
}

}  // namespace mla
