// Dense attention forward (FlashAttention style) for sm_103a (GB300).
//
// What it computes: for batch entry b, head h and query i < S, scaled-dot-
// product attention over keys t < S (t <= i when causal):
//   s_t = scale * q[b][i][h] . k[b][t][h]          (d_qk dims)
//   out[b][i][h] = sum_t softmax(s)_t v[b][t][h]  (d_v dims, bf16)
//   lse[b][h][i] = ln sum_t exp(s_t)               (fp32)
// The pages name FlashAttention without a formula: the TileLang talk
// ("Tile级原语与自动推理机制融合，TileAI社区发起人深度剖析TileLang核心技术与优势",
// performance section: MLA, FlashAttention and block-sparse kernels on par
// with CUTLASS) and the GEMM tutorial summary ("Designing high-performance
// GPU kernels with TileLang: Tensor-Core GEMM", key capabilities: fused GEMM
// + softmax that keeps the scores out of HBM).  DeepSeek's MLA prefill runs
// this form with 128 heads, d_qk = 192 (128 + 64 rotary) and d_v = 128.
//
// GB300 design:
//  * Persistent: one CTA per SM, each taking every grid-th work item, a
//    work item being a (128-query tile, head, batch entry).  Items are
//    ordered in chunks of 16 (batch, head) pairs so that the items running
//    at one time share the K/V of a few heads in L2; within a chunk a causal
//    grid takes the longest tiles first.  The roles count K/V tiles across
//    items, so the loads, score MMAs and softmax of one item overlap the
//    tail of the one before (set-up, Q and the first K/V tiles are no
//    longer paid per item).  Warp 0 issues the TMA loads of Q (per item) and
//    of the K tiles, warp 2 those of the V tiles (128 keys each, two-deep
//    rings of their own), so a K tile never waits behind a V tile; warp 1
//    owns TMEM and issues the MMAs; warps 4-11 run the softmax and the
//    epilogue with two threads per query row, 64 key columns each (warp w
//    reaches 16 lanes of TMEM lane quadrant w % 4 through the 16x32bx2
//    access shape).
//  * S = Q K^T (M=128, N=128, K=d_qk) takes Q from TMEM and K (K-major)
//    from shared memory and lands in one of two 128-column TMEM tiles.  Q is
//    staged in shared memory by the TMA while the previous item runs and
//    copied into TMEM with tcgen05.cp (in order with the MMAs) once that
//    item's last score MMA is done.  The softmax writes P as bf16 over the
//    first 64 columns of the score tile, and P.V reads P from TMEM as its A
//    operand with V as the MN-major B operand: P never goes through shared
//    memory, O (d_v fp32 columns) stays in TMEM until the epilogue, which
//    writes each row's 128 bytes per thread as 32-byte stores.
//  * The MMAs are issued in the order S(j), P.V(j-1): the score MMA of the
//    next tile runs on the tensor pipe while this tile's softmax computes;
//    an item's last P.V goes out right after its probabilities.
//  * Online softmax in the log2 domain with a lazy rescale: O and the sums
//    are rescaled only when a row max grows by more than 2^8, and the final
//    1/l and lse use the same reference max, so the result is exact.  out is
//    normalised by the sum of the bf16 probabilities P.V multiplies, which
//    the tensor core accumulates beside O: the P.V MMA runs with N = d_v +
//    16, its B operand the V tile followed by a box of bf16 ones (one MMA
//    per K step instead of a second, tiny one); lse comes from the softmax
//    threads' fp32 sum.
//  * Every wait is bounded (2 s on %globaltimer): on expiry the kernel
//    records MLA_ERR_DEVICE_TIMEOUT, lets in-flight copies and MMAs land,
//    frees TMEM and returns.
#include <cuda.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <mutex>

#include "mla.h"
#include "mla_internal.h"
#include "ptx_sm103.cuh"

namespace mla {
namespace {

constexpr int kAttThreads = 384;
constexpr int kSoftWarp0 = 4;                 // warps 4-11: softmax and epilogue
constexpr int kSoftWarps = 8;                 // two per TMEM lane quadrant, 16 rows each
constexpr int kTQ = 128, kTK = 128;           // query rows and keys per tile
constexpr int kAttDv = 128;
constexpr int kMaxDqkBoxes = 3;               // d_qk <= 192
constexpr int kChunk = 16;                    // (batch, head) pairs whose blocks run together
constexpr uint32_t kBox = 16384;              // 128 rows x 64 bf16, 128-byte swizzle
// Shared memory in 14 units of one box.  P.V runs with N = d_v + 16: the B
// operand is the V tile (two 64-dim boxes) followed by a box of bf16 ones,
// so the same MMA also accumulates each row's sum of P beside O.  An
// M/N-major operand's 64-column boxes sit one stride (LBO) apart, so the
// ones box lies two strides past each V stage's first box: stage 0's boxes
// are units 11 and 12 (stride 1), stage 1's units 7 and 10 (stride 3), the
// ones unit 13.  Q takes units 0-2 and the K stages the rest (each K step
// addresses its box on its own).
constexpr uint32_t kSQ = 0;
__host__ __device__ constexpr uint32_t k_box(int s, int c) {
  return (s == 0 ? 3u + (uint32_t)c : (c == 0 ? 6u : 7u + (uint32_t)c)) * kBox;
}
__host__ __device__ constexpr uint32_t v_box(int s, int c) {
  return (s == 0 ? 11u + (uint32_t)c : (c == 0 ? 7u : 10u)) * kBox;
}
__host__ __device__ constexpr uint32_t v_lbo(int s) { return s == 0 ? kBox : 3u * kBox; }
constexpr uint32_t kSOnes = 13 * kBox;
constexpr uint32_t kOnesBytes = kBox;
static_assert(v_box(0, 0) + 2 * v_lbo(0) == kSOnes && v_box(1, 0) + 2 * v_lbo(1) == kSOnes,
              "the ones box follows each V stage at two strides");
static_assert(v_box(0, 1) == v_box(0, 0) + v_lbo(0) && v_box(1, 1) == v_box(1, 0) + v_lbo(1),
              "V boxes one stride apart");
constexpr uint32_t kABar = 14 * kBox;
enum ABar : int {
  A_QFULL = 0,
  A_KFULL = 1,     // [2]
  A_KEMPTY = 3,    // [2]
  A_VFULL = 5,     // [2]
  A_VEMPTY = 7,    // [2]
  A_SFULL = 9,     // [2] score tile ready (MMA commit)
  A_PFULL = 11,    // [2] P written over the tile, O rescaled if needed (8 softmax warps)
  A_ODONE = 13,    // one phase per P.V MMA group
  A_QEMPTY = 14,   // the item's Q has been copied into TMEM: its staging buffer may be reloaded
  A_SDONE = 15,    // the item's last score MMA is done: Q's TMEM columns may be rewritten
  A_COUNT = 16
};
constexpr uint32_t kAMisc = kABar + 8 * 16;
constexpr uint32_t kASmem = kAMisc + 16 + 1024;
// TMEM: two score tiles, O and the P sums (one P.V result), and Q (the A
// operand of the score MMAs, d_qk / 2 columns of bf16 pairs)
constexpr uint32_t kColS = 0, kColO = 256, kColL = 384, kColQ = 400, kATmemCols = 512;
static_assert(kColQ + kMaxDqkBoxes * 64 / 2 <= kATmemCols, "Q fits beside O");
constexpr int kSumCols = 16;                  // P.1: every column holds the row's sum
static_assert(kColL == kColO + kAttDv, "the P sums are the last 16 columns of the P.V result");
constexpr float kARescale = 8.0f;
constexpr float kALn2 = 0.69314718055994530942f;
constexpr uint64_t kAWaitNs = 2000000000ull;
constexpr uint64_t kADrainNs = 2000000ull;
static_assert(kASmem <= 232448, "shared memory");

struct AttArgs {
  void* out;       // bf16 [B, S, H, d_v]
  float* lse;      // fp32 [B, H, S]
  int B, S, H, dqk, causal, n_qt;
  int out_v8;      // out is 32-byte aligned: each thread's 128 bytes go out as four 32-byte stores
  float scale_log2;
  int* err;
};

struct ACtx {
  uint32_t sbase, abort_addr;
  int* err;
  __device__ __forceinline__ uint32_t bar(int i) const { return sbase + kABar + 8u * i; }
};

__device__ __forceinline__ bool await_(const ACtx& x, uint32_t bar, uint32_t parity) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = ptx::globaltimer();
  for (uint32_t i = 1;; ++i) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    if ((i & 63u) == 0u) {
      if (ptx::ld_shared_u32_volatile(x.abort_addr) != 0u) return false;
      if (ptx::globaltimer() - t0 > kAWaitNs) {
        atomicCAS(x.err, 0, MLA_ERR_DEVICE_TIMEOUT);
        ptx::st_shared_u32(x.abort_addr, 1u);
        return false;
      }
    }
  }
}
__device__ __forceinline__ bool await_warp(const ACtx& x, uint32_t bar, uint32_t parity) {
  return __all_sync(0xffffffffu, await_(x, bar, parity));
}

// Work item `item` (a 128-query tile of one head of one batch entry).  Items
// run in chunks of kChunk (batch, head) pairs, and within a chunk the
// heaviest (last) query tiles of its pairs come first: the items running at
// one time then share the K/V of a few heads, which stay in L2 (all heads at
// once would stream K/V from HBM once per query tile).
struct AItem {
  int b, h, qt, n_kt;
};
__device__ __forceinline__ AItem att_item(const AttArgs& a, int item) {
  const int bh_n = a.B * a.H;
  const int chunk = item / (kChunk * a.n_qt);
  const int in_chunk = item - chunk * kChunk * a.n_qt;
  const int width = min(kChunk, bh_n - chunk * kChunk);
  const int rank = in_chunk / width;
  const int bh = chunk * kChunk + in_chunk % width;
  AItem it;
  it.qt = a.causal ? a.n_qt - 1 - rank : rank;
  it.b = bh / a.H;
  it.h = bh % a.H;
  it.n_kt = a.causal ? it.qt + 1 : (a.S + kTK - 1) / kTK;
  return it;
}

__global__ void __launch_bounds__(kAttThreads, 1)
    mla_attention_kernel(const __grid_constant__ CUtensorMap tm_q,
                         const __grid_constant__ CUtensorMap tm_k,
                         const __grid_constant__ CUtensorMap tm_v, const AttArgs args) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  ACtx x;
  x.sbase = (ptx::smem_addr(smem_raw) + 1023u) & ~1023u;
  x.abort_addr = x.sbase + kAMisc + 4;
  x.err = args.err;
  const uint32_t tslot = x.sbase + kAMisc;

  const int nbq = args.dqk / 64;
  const int total_items = args.n_qt * args.B * args.H;

  if (threadIdx.x == 0) {
    ptx::mbar_init(x.bar(A_QFULL), 1);
    ptx::mbar_init(x.bar(A_QEMPTY), 1);
    for (int s = 0; s < 2; ++s) {
      ptx::mbar_init(x.bar(A_KFULL + s), 1);
      ptx::mbar_init(x.bar(A_KEMPTY + s), 1);
      ptx::mbar_init(x.bar(A_VFULL + s), 1);
      ptx::mbar_init(x.bar(A_VEMPTY + s), 1);
      ptx::mbar_init(x.bar(A_SFULL + s), 1);
      ptx::mbar_init(x.bar(A_PFULL + s), kSoftWarps);
    }
    ptx::mbar_init(x.bar(A_ODONE), 1);
    ptx::mbar_init(x.bar(A_SDONE), 1);
    ptx::st_shared_u32(x.abort_addr, 0u);
    ptx::fence_mbarrier_init();
  }
  for (uint32_t o = threadIdx.x * 16u; o < kOnesBytes; o += kAttThreads * 16u)
    ptx::st_shared_v4(x.sbase + kSOnes + o, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u);
  ptx::fence_proxy_async_smem();   // the tensor core reads them
  if (warp == 1) {
    ptx::tmem_alloc(tslot, kATmemCols);
    ptx::tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    ptx::prefetch_tmap(&tm_q);
    ptx::prefetch_tmap(&tm_k);
    ptx::prefetch_tmap(&tm_v);
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = ptx::ld_shared_u32_volatile(tslot);

  // Every role walks the same items (item = blockIdx.x + k * gridDim.x) and
  // counts K/V tiles across them (jt): stage, score tile and barrier phases
  // follow jt, so one item's tail overlaps the next one's head.
  if (warp == 0 || warp == 2) {
    // Two producer threads: warp 0 loads Q and the K tiles, warp 2 the V
    // tiles, so that a K tile goes out as soon as its stage is free (its
    // score MMA two tiles back) and never waits behind a V tile (whose stage
    // is freed later, by a P.V).
    const bool kq = (warp == 0);
    if (lane == 0) {
      uint32_t jt = 0, nq = 0;
      bool ok = true;
      auto load_k = [&](const AItem& it, int j) -> bool {
        const int s = (int)(jt & 1u);
        const uint32_t ph = (jt >> 1) & 1u;
        if (!await_(x, x.bar(A_KEMPTY + s), ph ^ 1u)) return false;
        ptx::mbar_arrive_expect_tx(x.bar(A_KFULL + s), nbq * kBox);
        for (int c = 0; c < nbq; ++c)
          ptx::tma_load_4d(x.sbase + k_box(s, c), &tm_k, 64 * c, it.h,
                           j * kTK, it.b, x.bar(A_KFULL + s));
        return true;
      };
      auto load_v = [&](const AItem& it, int j) -> bool {
        const int s = (int)(jt & 1u);
        const uint32_t ph = (jt >> 1) & 1u;
        if (!await_(x, x.bar(A_VEMPTY + s), ph ^ 1u)) return false;
        ptx::mbar_arrive_expect_tx(x.bar(A_VFULL + s), 2 * kBox);
        for (int c = 0; c < 2; ++c)
          ptx::tma_load_4d(x.sbase + v_box(s, c), &tm_v, 64 * c, it.h, j * kTK, it.b,
                           x.bar(A_VFULL + s));
        return true;
      };
      for (int item = (int)blockIdx.x; ok && item < total_items; item += (int)gridDim.x) {
        const AItem it = att_item(args, item);
        if (!kq) {
          for (int j = 0; ok && j < it.n_kt; ++j, ++jt) ok = load_v(it, j);
          continue;
        }
        // the item's first K tile (its stage is freed by the score MMA two
        // tiles back), then Q (once the previous item's Q has been copied
        // into TMEM), then the rest in tile order
        ok = load_k(it, 0);
        if (!ok) break;
        if (!await_(x, x.bar(A_QEMPTY), (nq & 1u) ^ 1u)) break;
        ptx::mbar_arrive_expect_tx(x.bar(A_QFULL), nbq * kBox);
        for (int c = 0; c < nbq; ++c)
          ptx::tma_load_4d(x.sbase + kSQ + c * kBox, &tm_q, 64 * c, it.h, it.qt * kTQ, it.b,
                           x.bar(A_QFULL));
        ++nq;
        ++jt;
        for (int j = 1; ok && j < it.n_kt; ++j, ++jt) ok = load_k(it, j);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // S(t) = Q K(t)^T, then P(t-1).V(t-1) (+ P(t-1).1) within an item; an
    // item's last P.V follows its last score MMA
    constexpr uint32_t id_s = ptx::idesc_f32acc(kTQ, kTK, 0, 0, 1);
    // P.V and P.1 in one MMA: N = d_v + 16 (V's columns, then the ones box)
    constexpr uint32_t id_o = ptx::idesc_f32acc(kTQ, kAttDv + kSumCols, 0, 1, 1);
    auto issue_pv = [&](uint32_t tt, bool first) -> bool {
      const int s = (int)(tt & 1u);
      const uint32_t ph = (tt >> 1) & 1u;
      if (!await_warp(x, x.bar(A_PFULL + s), ph)) return false;
      if (!await_warp(x, x.bar(A_VFULL + s), ph)) return false;
      ptx::tc_fence_after();
#pragma unroll
      for (int k = 0; k < kTK / 16; ++k) {
        // B: the stage's two V boxes and the ones box, one stride (LBO)
        // apart along N; 8-key groups 1 KB apart, a K step 16 keys (2 KB).
        // The last 16 result columns are the sums of the bf16 probabilities
        // P.V multiplies, accumulated (and rescaled) beside O.
        const uint64_t bd = ptx::smem_desc(x.sbase + v_box(s, 0) + k * 2048, v_lbo(s), 1024,
                                           ptx::kLayoutSw128);
        ptx::mma_ts_elect(tmem + kColO, tmem + kColS + 128u * s + 8u * k, bd, id_o,
                          (!first || k > 0) ? 1u : 0u);
      }
      ptx::mma_commit_elect(x.bar(A_VEMPTY + s));
      ptx::mma_commit_elect(x.bar(A_ODONE));
      return true;
    };
    uint32_t jt = 0, nq = 0;
    bool ok = true, pending = false, pending_first = false;
    uint32_t pending_t = 0;
    for (int item = (int)blockIdx.x; ok && item < total_items; item += (int)gridDim.x) {
      const AItem it = att_item(args, item);
      // The item's Q: staged in shared memory by the TMA (loaded while the
      // previous item ran), copied into TMEM once the previous item's last
      // score MMA is done; the staging buffer is free once the copy is.
      if (!await_warp(x, x.bar(A_QFULL), nq & 1u)) {
        ok = false;
        break;
      }
      if (nq > 0 && !await_warp(x, x.bar(A_SDONE), (nq - 1) & 1u)) {
        ok = false;
        break;
      }
      ++nq;
      ptx::tc_fence_after();
      for (int k = 0; k < nbq * 4; ++k)
        ptx::tmem_cp_128x256b_elect(
            tmem + kColQ + 8u * (uint32_t)k,
            ptx::smem_desc(x.sbase + kSQ + (uint32_t)(k >> 2) * kBox + (uint32_t)(k & 3) * 32u, 16,
                           1024, ptx::kLayoutSw128));
      ptx::mma_commit_elect(x.bar(A_QEMPTY));
      for (int j = 0; j < it.n_kt; ++j, ++jt) {
        const int s = (int)(jt & 1u);
        const uint32_t ph = (jt >> 1) & 1u;
        if (!await_warp(x, x.bar(A_KFULL + s), ph)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        for (int k = 0; k < nbq * 4; ++k) {
          // A = Q from TMEM (a K step of 16 dims is 8 columns), B = the K box
          const uint64_t bd = ptx::smem_desc(x.sbase + k_box(s, k >> 2) + (uint32_t)(k & 3) * 32u, 16,
                                             1024, ptx::kLayoutSw128);
          ptx::mma_ts_elect(tmem + kColS + 128u * s, tmem + kColQ + 8u * (uint32_t)k, bd, id_s,
                            k ? 1u : 0u);
        }
        ptx::mma_commit_elect(x.bar(A_SFULL + s));
        ptx::mma_commit_elect(x.bar(A_KEMPTY + s));
        if (j == it.n_kt - 1) ptx::mma_commit_elect(x.bar(A_SDONE));   // Q's columns may be rewritten
        if (pending && !issue_pv(pending_t, pending_first)) {
          ok = false;
          break;
        }
        pending = true;
        pending_t = jt;
        pending_first = (j == 0);
      }
      // the item's last P.V right away: the epilogue waits for it, and the
      // next item's first score MMA would otherwise go ahead of it
      if (ok && pending) {
        ok = issue_pv(pending_t, pending_first);
        pending = false;
      }
    }
    __syncwarp();
  } else if (warp >= kSoftWarp0) {
    // Two threads per query row: warp w works on 16 lanes (the first or the
    // second 16) of TMEM lane quadrant w % 4; lane t takes lane t & 15 of
    // them and key columns [64 (t >> 4), +64) of each tile.
    const int sw = warp - kSoftWarp0;
    const int quad = warp & 3;
    const int sub = sw >> 2;
    const int half = lane >> 4;
    const int r = quad * 32 + sub * 16 + (lane & 15);
    const uint32_t lanes = (uint32_t)(quad * 32 + sub * 16) << 16;
    const float sl2 = args.scale_log2;
    uint32_t jt = 0;
    bool ok = true;
    AItem nit = att_item(args, (int)blockIdx.x);
    for (int item = (int)blockIdx.x; ok && item < total_items; item += (int)gridDim.x) {
      const AItem it = nit;
      const int qi = it.qt * kTQ + r;
      float m_ref = -INFINITY, l_f = 0.f;   // fp32 sum of this thread's columns (for lse)
      for (int j = 0; j < it.n_kt; ++j, ++jt) {
        const int s = (int)(jt & 1u);
        if (!await_warp(x, x.bar(A_SFULL + s), (jt >> 1) & 1u)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        float sv[64];
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t v[32];
          ptx::tmem_ld16x2_wait<64>(tmem + lanes + kColS + 128u * s + 32u * c, v);
#pragma unroll
          for (int k = 0; k < 32; ++k) sv[32 * c + k] = __uint_as_float(v[k]);
        }
        // keys past the sequence, or after the query when causal, get no weight
        const int k0 = j * kTK + 64 * half;
        const int lim = args.causal ? min(qi + 1, args.S) : args.S;
        if (__any_sync(0xffffffffu, k0 + 64 > lim)) {
#pragma unroll
          for (int k = 0; k < 64; ++k)
            if (k0 + k >= lim) sv[k] = -INFINITY;
        }
        float m4[4];
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          const float* a = sv + 16 * q4;
          m4[q4] = ptx::max3(ptx::max3(ptx::max3(a[0], a[1], a[2]), ptx::max3(a[3], a[4], a[5]),
                                       ptx::max3(a[6], a[7], a[8])),
                             ptx::max3(a[9], a[10], a[11]), ptx::max3(a[12], a[13], fmaxf(a[14], a[15])));
        }
        float mx = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));   // the row's other half
        const float m_cand = fmaxf(m_ref, mx * sl2);
        const bool rescale = (j > 0) && (m_cand > m_ref + kARescale);
        float alpha = 1.0f;
        if (j == 0) {
          m_ref = m_cand;
        } else if (rescale) {
          alpha = ptx::ex2(m_ref - m_cand);
          m_ref = m_cand;
          l_f *= alpha;
        }
        const float neg_m = (m_ref == -INFINITY) ? 0.f : -m_ref;
        uint32_t pk[32];
        const uint64_t sc2 = ptx::f2_pack(sl2, sl2);
        const uint64_t nm2 = ptx::f2_pack(neg_m, neg_m);
        uint64_t sf2[2] = {0ull, 0ull};
#pragma unroll
        for (int k = 0; k < 32; ++k) {
          float xa, xc;
          ptx::f2_unpack(ptx::f2_fma(ptx::f2_pack(sv[2 * k], sv[2 * k + 1]), sc2, nm2), xa, xc);
          const float a = ptx::ex2(xa), c = ptx::ex2(xc);
          sf2[k & 1] = ptx::f2_add(sf2[k & 1], ptx::f2_pack(a, c));
          pk[k] = ptx::pack_bf16x2(a, c);
        }
        {
          float fa, fc;
          ptx::f2_unpack(ptx::f2_add(sf2[0], sf2[1]), fa, fc);
          l_f += fa + fc;
        }
        // P (bf16 pairs) over the first 64 columns of the score tile: this
        // thread's 64 keys are packed columns [32 half, +32)
        ptx::tmem_st16x2<32>(tmem + lanes + kColS + 128u * s, pk);
        ptx::tmem_wait_st();
        // O must not be rescaled before the previous P.V has landed (waited
        // on every tile but an item's first, which keeps the phase of the
        // P.V barrier within one of this wait's parity)
        if (j > 0 && !await_warp(x, x.bar(A_ODONE), (jt - 1) & 1u)) {
          ok = false;
          break;
        }
        if (__any_sync(0xffffffffu, rescale)) {
          ptx::tc_fence_after();
#pragma unroll 1
          for (int c = 0; c < 2; ++c) {
            uint32_t o[32];
            ptx::tmem_ld16x2_wait<64>(tmem + lanes + kColO + 32u * c, o);
#pragma unroll
            for (int k = 0; k < 32; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * alpha);
            ptx::tmem_st16x2<64>(tmem + lanes + kColO + 32u * c, o);
          }
          {
            uint32_t l8[8];   // the row's P sums, 8 of the 16 columns per thread
            ptx::tmem_ld16x2_x8_wait<8>(tmem + lanes + kColL, l8);
#pragma unroll
            for (int k = 0; k < 8; ++k) l8[k] = __float_as_uint(__uint_as_float(l8[k]) * alpha);
            ptx::tmem_st16x2_x8<8>(tmem + lanes + kColL, l8);
          }
          ptx::tmem_wait_st();
        }
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(x.bar(A_PFULL + s));
      }
      if (!ok) break;
      // Epilogue: O / l and lse once the item's last P.V has landed; each
      // thread writes its 64 of the row's 128 output dims.  The next item's
      // first P.V (which overwrites O) waits for this item's P of its first
      // tile, which these threads write only after this.
      l_f += __shfl_xor_sync(0xffffffffu, l_f, 16);
      // the next item's coordinates (integer divisions), while the last P.V
      // runs
      if (item + (int)gridDim.x < total_items) nit = att_item(args, item + (int)gridDim.x);
      if (!await_warp(x, x.bar(A_ODONE), (jt - 1) & 1u)) {
        ok = false;
        break;
      }
      ptx::tc_fence_after();
      uint32_t l8[8];
      ptx::tmem_ld16x2_x8_wait<8>(tmem + lanes + kColL, l8);
      const float l_b = __uint_as_float(l8[0]);
      const float inv_l = l_b > 0.f ? 1.0f / l_b : 0.f;
      const bool valid = qi < args.S;
      uint16_t* orow = static_cast<uint16_t*>(args.out) +
                       (((int64_t)it.b * args.S + (valid ? qi : 0)) * args.H + it.h) * kAttDv + 64 * half;
      // this thread's 64 output dims as bf16 pairs, then out in 32-byte (or
      // 16-byte) stores: a warp's rows lie H * d_v apart in memory, so whole
      // sectors per store is what keeps the epilogue short
      uint32_t pk[32];
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint32_t o[32];
        ptx::tmem_ld16x2_wait<64>(tmem + lanes + kColO + 32u * c, o);
#pragma unroll
        for (int k = 0; k < 16; ++k)
          pk[16 * c + k] =
              ptx::pack_bf16x2(__uint_as_float(o[2 * k]) * inv_l, __uint_as_float(o[2 * k + 1]) * inv_l);
      }
      if (valid) {
        if (args.out_v8) {
#pragma unroll
          for (int q = 0; q < 4; ++q)
            ptx::st_global_v8(orow + 16 * q, pk[8 * q], pk[8 * q + 1], pk[8 * q + 2], pk[8 * q + 3],
                              pk[8 * q + 4], pk[8 * q + 5], pk[8 * q + 6], pk[8 * q + 7]);
        } else {
          uint4* dst = reinterpret_cast<uint4*>(orow);
#pragma unroll
          for (int q = 0; q < 8; ++q)
            dst[q] = make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
        }
      }
      if (valid && half == 0)
        args.lse[((int64_t)it.b * args.H + it.h) * args.S + qi] =
            l_f > 0.f ? (m_ref + log2f(l_f)) * kALn2 : -INFINITY;
      ptx::tc_fence_before();
    }
  }
  __syncthreads();
  if (ptx::ld_shared_u32_volatile(x.abort_addr) != 0u) {
    const uint64_t t0 = ptx::globaltimer();
    while (ptx::globaltimer() - t0 < kADrainNs) __nanosleep(1000);
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kATmemCols);
  }
}

std::once_flag g_att_once[64];
cudaError_t g_att_status[64];

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace mla

using namespace mla;

extern "C" int mla_attention_fwd(const void* q, const void* k, const void* v, void* out,
                                 float* lse, int batch, int seqlen, int heads, int d_qk, int d_v,
                                 int causal, float softmax_scale, void* stream) {
  if (!q || !k || !v || !out || !lse || batch < 1 || seqlen < 1 || heads < 1 ||
      (d_qk != 64 && d_qk != 128 && d_qk != 192) || d_v != kAttDv || !(softmax_scale > 0.f) ||
      !isfinite(softmax_scale) || !aligned16(q) || !aligned16(k) || !aligned16(v) ||
      !aligned16(out) || (reinterpret_cast<uintptr_t>(lse) & 3u))
    return MLA_ERR_INVALID_ARG;
  const long long n_qt = (seqlen + kTQ - 1) / kTQ;
  const long long grid = n_qt * batch * heads;
  if (grid >= (1ll << 31) || (long long)batch * seqlen * heads * d_qk >= (1ll << 40))
    return MLA_ERR_INVALID_ARG;
  int device = 0, sms = 0;
  int* err = nullptr;
  const int st = device_current(&device, &sms, &err);
  if (st != MLA_OK) return st;
  if (device < 0 || device >= 64) return MLA_ERR_INVALID_ARG;
  std::call_once(g_att_once[device], [&]() {
    g_att_status[device] = cudaFuncSetAttribute(
        mla_attention_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kASmem);
  });
  if (g_att_status[device] != cudaSuccess) return MLA_ERR_CUDA;
  CUtensorMap mq, mk, mv;
  const uint64_t dqk4[4] = {(uint64_t)d_qk, (uint64_t)heads, (uint64_t)seqlen, (uint64_t)batch};
  const uint64_t sqk[3] = {(uint64_t)d_qk * 2, (uint64_t)heads * d_qk * 2,
                           (uint64_t)seqlen * heads * d_qk * 2};
  const uint64_t dv4[4] = {(uint64_t)d_v, (uint64_t)heads, (uint64_t)seqlen, (uint64_t)batch};
  const uint64_t sv[3] = {(uint64_t)d_v * 2, (uint64_t)heads * d_v * 2,
                          (uint64_t)seqlen * heads * d_v * 2};
  const uint32_t box[4] = {64, 1, kTQ, 1};
  if (!encode_tiled_map(&mq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, q, dqk4, sqk, box,
                        CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_tiled_map(&mk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, k, dqk4, sqk, box,
                        CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_tiled_map(&mv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, v, dv4, sv, box,
                        CU_TENSOR_MAP_SWIZZLE_128B))
    return MLA_ERR_CUDA;
  AttArgs a;
  a.out = out;
  a.lse = lse;
  a.B = batch;
  a.S = seqlen;
  a.H = heads;
  a.dqk = d_qk;
  a.causal = causal ? 1 : 0;
  a.n_qt = (int)n_qt;
  a.out_v8 = (reinterpret_cast<uintptr_t>(out) & 31u) == 0 ? 1 : 0;
  a.scale_log2 = softmax_scale * 1.4426950408889634f;
  a.err = err;
  // persistent: one CTA per SM, each taking every grid-th work item
  const unsigned ctas = (unsigned)(grid < (long long)sms ? grid : (long long)sms);
  mla_attention_kernel<<<ctas, kAttThreads, kASmem, static_cast<cudaStream_t>(stream)>>>(
      mq, mk, mv, a);
  return cudaGetLastError() == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}
