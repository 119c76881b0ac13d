// Paged MLA decode, main kernel, for sm_103a (GB300).
//
// What it computes: for each query row (batch b, query token i, head h),
// softmax(scale * q . k_t) weighted sum of the first 512 dims of the visible
// latent cache rows k_t, plus the log-sum-exp, over the pages assigned to this
// cluster by the split-KV plan.  This is the DeepSeek MLA / FlashMLA decode
// kernel that the TileLang talk walks through ("Tile级原语与自动推理机制融合，
// TileAI社区发起人深度剖析TileLang核心技术与优势", section 什么是「TileLang」);
// its online-softmax row max is the "accum_s -> scores_max" reduce whose
// layout follows from the GEMM that produces accum_s (same section, step 2 of
// layout inference): here that GEMM is a tcgen05 MMA with a 128-lane TMEM
// accumulator, so one thread owns one row and the reduce is a per-thread loop.
// As the talk's pipeline section says, only copies and GEMMs are truly
// asynchronous, and the copies get their own pipeline stage: here a TMA
// producer warp streams 64-token pages through an mbarrier ring.
//
// GB300 design (not the talk's):
//  * One work unit is a cluster of two CTAs on two SMs.  A 128-row tile of
//    queries has an fp32 output of 128 x 512 = all 512 TMEM columns of one SM,
//    so CTA r owns output dims [256 r, 256 r + 256) for all 128 rows.
//  * The 576-wide Q.K^T reduction is split between the CTAs as well: CTA r
//    multiplies its latent half (dims [256 r, 256 r + 256)) plus half of the
//    rotary dims ([512 + 32 r, 512 + 32 r + 32)).  Each CTA therefore loads
//    exactly 36 KB of every 72 KB page: the pair reads each page once, with
//    no duplicated tensor work.
//  * The softmax is split by rows: CTA r owns 16 rows of every TMEM lane
//    quadrant (lanes 32 q + 16 r + [0, 16)), 64 in all.  For every page it
//    sends the peer the 64 x 64 partial scores of the peer's rows (12 KB:
//    fp32 rounded to 24-bit floats, relative error <= 2^-16, within what the
//    fp32 accumulation of the 288 products already allows; st.async), adds
//    the peer's partial for its own rows, runs the
//    online softmax for them and sends back their bf16 probabilities and
//    rescale factors (8 KB, TMA bulk copies), so both CTAs hold P for all 128
//    rows for their halves of O.  All cross-SM traffic goes into the peer's
//    shared memory and completes on its mbarriers.  Distributed shared memory
//    moves only about 40 GB/s out of each SM on GB300, and these transfers
//    (about 20 KB each way per page) are what bounds the page rate; sending
//    the whole 32 KB partial tile both ways would be worse.
//  * Page workers: warps 0-3 take the even pages of the CTA's work and warps
//    4-7 the odd ones, warp q of a set working on lane quadrant q (its 16
//    owned rows, two threads per row through the 16x32bx2 TMEM access shape,
//    and its 16 peer rows).  A worker ships its page's partial scores, runs
//    the softmax, copies out its probabilities and imports the peer's; the
//    running row max passes from one page's worker to the next through
//    shared memory and an mbarrier, so the online softmax stays sequential
//    while two pages' chains of waits overlap.  Warp 8 is the TMA producer,
//    warp 9 issues the score MMAs and owns TMEM, warp 11 issues the P.V MMAs
//    (each from one elected lane of a converged warp), and one thread of
//    warp 10 tells the peer when a P buffer is free.
//  * A thread that has a remote operation in flight (a copy or an arrive on
//    the peer's barrier) does not also signal the local barriers of the
//    critical path: a release arrive may wait for that remote operation to
//    complete, which the transfers queued ahead of it make slow.
//  * S = Q K^T: M=128, N=64, 18 K-steps (16 latent with Q read from TMEM, 2
//    rotary from shared memory) into a double buffered TMEM score tile;
//    O += P V: M=128, N=256, K=64 with P from shared memory and V from the
//    same shared-memory page as K (as an MN-major operand).
//  * Online softmax in the log2 domain with a lazy rescale: O is rescaled only
//    when the row max grows by more than 2^8; the final 1/l and lse use the
//    same (possibly stale) max, so the result is exact.
//  * Every wait is bounded (globaltimer); on expiry the kernel records
//    MLA_ERR_DEVICE_TIMEOUT, tells the peer CTA, lets in-flight copies land,
//    frees TMEM and returns.  No trap, no unbounded spin.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <limits.h>
#include <math.h>
#include <stdint.h>

#include "mla.h"
#include "mla_internal.h"
#include "ptx_sm103.cuh"

namespace mla {
namespace {

// Warp roles (see above).  Warp w reaches TMEM lanes [32 (w % 4), +32).
constexpr int kThreads = 480;         // launched for sparse decode
constexpr int kDenseThreads = 384;    // dense decode: warps 0-11 only
constexpr int kQuadWarps = 4;   // page workers per set (one per TMEM lane quadrant)
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kPSendWarp = 10;   // the P notifier thread
constexpr int kPvWarp = 11;
constexpr int kGatherWarp = 12;   // sparse decode: warps 12-14 gather with warp 8 (idle when dense)
constexpr int kGatherWarps = 4;   // sparse decode: each gathers 64 / kGatherWarps rows of a chunk
constexpr int kGatherRows = 64 / kGatherWarps;
static_assert(kThreads == 32 * (kGatherWarp + kGatherWarps - 1), "gather warps end the block");
static_assert(kGatherRows % 8 == 0 && kGatherRows <= 32, "rotary copies take 8 rows at a time");
constexpr uint64_t kWaitTimeoutNs = 2000000000ull;   // 2 s per wait
constexpr uint64_t kDrainNs = 2000000ull;            // 2 ms settle time after an abort
constexpr float kRescaleThreshold = 8.0f;           // log2 units
constexpr float kLn2 = 0.69314718055994530942f;
constexpr int kHalfRows = 64;                        // softmax rows owned by one CTA
constexpr int kSubRows = 16;                         // of them in each TMEM lane quadrant
constexpr int kRemoteLane = 31;   // the lane that issues a warp's remote copies and arrives

// TMEM columns (fp32 / packed-bf16x2 32-bit cells, 128 lanes).
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 0;     // [0, 256): this CTA's half of O
constexpr uint32_t kColS = 256;   // two 64-column score tiles
constexpr uint32_t kColQ = 384;   // Q's latent half, bf16x2: 128 rows x 256 dims

// Shared memory (offsets from a 1024-byte aligned base).
constexpr int kStages = 4;
// Receive buffers for the peer's partial scores and P buffers: page g uses
// buffer g % 2, like its score tile and its worker set.
constexpr int kRBufs = 2;
constexpr int kPBufs = 2;
constexpr uint32_t kQRope = 0;            // [128 x 32] bf16, 64-byte swizzle
constexpr uint32_t kStage0 = 8192;        // kStages x 36 KB
constexpr uint32_t kStageBytes = 36864;
constexpr uint32_t kStageRope = 32768;    // rotary box inside a stage
// The peer's partial scores of my rows arrive as 24-bit floats, 64 columns =
// 192 bytes = 12 chunks of 16 bytes per row: [12 chunks][64 owned rows].
constexpr uint32_t kRecvChunks = 12;
constexpr uint32_t kRecv = kStage0 + kStages * kStageBytes;  // 2 x [12 chunks][64 owned rows] x 16 B
constexpr uint32_t kRecvBytes = kHalfRows * kRecvChunks * 16;
constexpr uint32_t kP = kRecv + kRBufs * kRecvBytes;  // kPBufs x [128 x 64] bf16, 128-byte swizzle
constexpr uint32_t kPBytes = 128 * 64 * 2;
constexpr uint32_t kAlphaBufBytes = 2 * kHalfRows * 4;
constexpr uint32_t kAlpha = kP + kPBufs * kPBytes;   // float[kPBufs][owner rank][64] rescale factors
constexpr uint32_t kInvL = kAlpha + kPBufs * kAlphaBufBytes;   // float[2 parities][owner rank][64] 1/l
constexpr uint32_t kHand = kInvL + 2 * 128 * 4;   // float[2 sets][4 quadrants][16] running max
constexpr uint32_t kSums = kHand + 2 * 4 * 16 * 4;  // float[2 parities][4][32 lanes][3] set 1's sums
constexpr uint32_t kEpiInv = kSums + 2 * 4 * 32 * 12;   // float[128]: 1/l of each tile row, for set 1
constexpr uint32_t kBar = kEpiInv + 128 * 4;
constexpr uint32_t kMisc = kBar + 8 * 48;
constexpr uint32_t kSmemAlloc = kMisc + 64 + 1024;  // + slack for 1024-byte alignment
static_assert(kP % 1024 == 0 && kStage0 % 1024 == 0, "swizzled buffers need 1 KB alignment");
// Page g uses score tile, receive buffer and P buffer g % 2, and its worker
// set is g % 2: every per-page barrier is then used by one set, in order.
static_assert(kRBufs == 2 && kPBufs == 2, "buffers are paired with the page worker sets");
static_assert(kSmemAlloc <= 232448, "shared memory");

// Bytes moved per stage / per Q tile by one CTA.
constexpr uint32_t kStageTx = 4 * 8192 + 4096;   // 4 latent boxes + rotary half
constexpr uint32_t kQRopeTx = 8192;
constexpr uint32_t kPRecvTx = kHalfRows * 128 + kHalfRows * 4;   // the peer's 64 P rows + factors
constexpr uint32_t kInvLTx = kHalfRows * 4;                        // the peer's 64 values of 1/l

// [2] = one per buffer: page g uses score tile, receive buffer and P buffer
// g % 2.  "Workers" are the page's four workers (the set g % 2).
enum Bar : uint32_t {
  B_FULL = 0,                 // [kStages] stage loaded (TMA tx)
  B_EMPTY = kStages,          // [kStages] stage consumed (MMA commit)
  B_QFULL = 2 * kStages,      // Q tile ready: rotary half (TMA) + latent half (set 1's 4 warps)
  B_QEMPTY,                   // last score MMA of a tile done
  B_SFULL,                    // [2] score tile ready (MMA commit)
  B_SEMPTY = B_SFULL + 2,     // [2] score tile read (the page's 4 workers)
  B_PFULL = B_SEMPTY + 2,     // [2] all 128 rows of P in shared memory and O rescaled (4 workers x 2)
  B_PEMPTY = B_PFULL + 2,     // [2] P.V done (MMA commit)
  B_OFULL = B_PEMPTY + 2,
  B_OEMPTY,                   // both sets' 8 warps have drained their columns of O
  B_RFULL,                    // [2] the peer's partial scores for my rows (st.async tx)
  B_REMPTY = B_RFULL + 2,     // [2] the peer's workers have read what I sent (4 remote arrives)
  B_PRECV = B_REMPTY + 2,     // [2] the peer's P rows and rescale factors arrived (bulk-copy tx)
  B_PFREE = B_PRECV + 2,      // [2] the peer's P buffer may take my next rows (peer's P.V done)
  B_LRECV = B_PFREE + 2,      // [2] the peer's 1/l for its rows arrived (per tile parity)
  B_HAND = B_LRECV + 2,       // [2 sets][4 quadrants] running max of the set's page handed on
  B_SUMS = B_HAND + 8,        // [2] set 1's sums of a tile handed to set 0 (per tile parity)
  B_SUMSFREE = B_SUMS + 2,    // [2] set 0 has read them
  B_TEARDOWN = B_SUMSFREE + 2,
  B_EPI,                      // set 0 has published 1/l of the tile's rows (4 warps)
  B_COUNT,
};
static_assert(B_COUNT <= 48, "barrier space");

struct Ctx {
  uint32_t sbase;       // 1024-aligned shared base
  uint32_t tmem;        // TMEM base address
  uint32_t rank, peer;
  uint32_t abort_addr, peer_abort_addr;
  int* err;
  __device__ __forceinline__ uint32_t bar(uint32_t i) const { return sbase + kBar + 8u * i; }
};

__device__ __forceinline__ void abort_all(const Ctx& x) {
  atomicCAS(x.err, 0, MLA_ERR_DEVICE_TIMEOUT);
  ptx::st_shared_u32(x.abort_addr, 1u);
  ptx::st_cluster_u32(x.peer_abort_addr, 1u);
}

// Bounded wait for the phase with parity `parity` of mbarrier `bar`.
__device__ __forceinline__ bool wait_bar(const Ctx& x, uint32_t bar, uint32_t parity,
                                         bool cluster_scope = false) {
  if (cluster_scope ? ptx::mbar_try_wait_cluster(bar, parity) : ptx::mbar_try_wait(bar, parity))
    return true;
  const uint64_t t0 = ptx::globaltimer();
  for (uint32_t i = 1;; ++i) {
    if (cluster_scope ? ptx::mbar_try_wait_cluster(bar, parity) : ptx::mbar_try_wait(bar, parity))
      return true;
    if ((i & 63u) == 0u) {
      if (ptx::ld_shared_u32_volatile(x.abort_addr) != 0u) return false;
      if (ptx::globaltimer() - t0 > kWaitTimeoutNs) {
        abort_all(x);
        return false;
      }
    }
  }
}

// The same, decided for the whole warp: a lane that gives up makes every lane
// give up, so warp-collective tcgen05 instructions after it are never reached
// by part of a warp.
__device__ __forceinline__ bool wait_warp(const Ctx& x, uint32_t bar, uint32_t parity,
                                          bool cluster_scope = false) {
  const bool ok = wait_bar(x, bar, parity, cluster_scope);
  return __all_sync(0xffffffffu, ok);
}

struct Work {
  int tile, rows, b0, p0, b1, p1, split0, stotal;
  const int32_t* items;
};

// 32 consecutive TMEM columns of this warp's 32 lanes, loaded and waited on
// in one statement so no use of the registers can be scheduled before the
// wait.
__device__ __forceinline__ void tmem_load32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}

// ------------------------------------------------------------------ producer
__device__ __forceinline__ bool run_producer(const Ctx& x, const Work& w, const DecodeParams& prm,
                                             const CUtensorMap* tm_q_rope,
                                             const CUtensorMap* tm_kv_lat,
                                             const CUtensorMap* tm_kv_rope) {
  const uint64_t policy = ptx::policy_evict_first();
  SegIter it{w.b0, w.p0, w.b1, w.p1, w.items};
  int b, pb, pe;
  uint32_t g = 0, n_item = 0;
  const int32_t xq_lat = 256 * (int32_t)x.rank, xq_rope = 512 + 32 * (int32_t)x.rank;
  // The first page's block-table entry is read alongside the first batch
  // item (SegIter), not after it: the cluster's first segment starts at
  // (b0, p0).
  const int first_page = ((unsigned)w.b0 < (unsigned)prm.batch && (unsigned)w.p0 < (unsigned)prm.max_pages)
                             ? prm.block_table[(size_t)w.b0 * prm.max_pages + w.p0]
                             : -1;
  while (it.next(b, pb, pe)) {
    // Entries past max_pages are never read: a sequence longer than its
    // block-table row is reported and served from page 0.
    const int32_t* bt = prm.block_table + (size_t)b * prm.max_pages;
    int next_page = (g == 0 && b == w.b0 && pb == w.p0) ? first_page
                                                       : (pb < prm.max_pages ? bt[pb] : -1);
    if (!wait_bar(x, x.bar(B_QEMPTY), (n_item & 1u) ^ 1u)) return false;
    ptx::mbar_arrive_expect_tx(x.bar(B_QFULL), kQRopeTx);
    const int32_t row0 = b * w.rows + w.tile * kTileRows;
    ptx::tma_load_2d(x.sbase + kQRope, tm_q_rope, xq_rope, row0, x.bar(B_QFULL));
    for (int pg = pb; pg < pe; ++pg, ++g) {
      int page = next_page;
      if (pg + 1 < pe) next_page = pg + 1 < prm.max_pages ? bt[pg + 1] : -1;
      const uint32_t s = g % kStages, k = g / kStages;
      if (!wait_bar(x, x.bar(B_EMPTY + s), (k & 1u) ^ 1u)) return false;
      if ((unsigned)page >= (unsigned)prm.num_pages) {
        atomicCAS(x.err, 0, MLA_ERR_DEVICE_BOUNDS);
        page = 0;
      }
      ptx::mbar_arrive_expect_tx(x.bar(B_FULL + s), kStageTx);
      const int32_t y = page * kPageTokens;
      const uint32_t st = x.sbase + kStage0 + s * kStageBytes;
      for (int ch = 0; ch < 4; ++ch)
        ptx::tma_load_2d_hint(st + ch * 8192, tm_kv_lat, xq_lat + 64 * ch, y, x.bar(B_FULL + s),
                              policy);
      ptx::tma_load_2d_hint(st + kStageRope, tm_kv_rope, xq_rope, y, x.bar(B_FULL + s), policy);
    }
    ++n_item;
  }
  return true;
}

// Sparse decode (one query token per entry): step g's "page" is the chunk
// of listed positions [64 pg, 64 pg + 64) of entry b, whose cache rows are
// scattered.  The whole producer warp gathers a chunk's rows (this CTA's 256
// latent and 32 rotary dims of each) with 16-byte cp.async copies, straight
// into the layout the tiled loads give a stage: latent box k (dims 64 k ..)
// row r, 16-byte chunk c at k * 8192 + r * 128 + ((c ^ (r % 8)) << 4)
// (128-byte swizzle); the rotary box row r, chunk c at kStageRope + r * 64 +
// ((c ^ ((r / 2) % 4)) << 4) (64-byte swizzle).  One instruction copies one
// row's 512 latent bytes (lane = chunk), so each is four whole 128-byte
// lines; eight more copy the rotary parts of eight rows each.  Rows past the
// entry's count are zero-filled (the copy form with a source size); listed
// rows use the plain 16-byte form, which retires faster, with an L2
// evict-first policy (each row is read once).
//
// The row each lane resolves (rows lane and lane + 32: list position, then
// block-table entry) is ready one chunk ahead, and the list positions two
// chunks ahead, so no dependent global load sits between two chunks' copies.
// Step g's copies are waited for once step g + kGatherLag is issued (all of
// them at the end of a tile, so that the next tile's Q wait cannot hold back
// the last score MMAs), then fenced to the async proxy and announced on the
// stage's FULL barrier.  kGatherLag < kStages: a stage the warp waits to
// refill was announced before.
constexpr uint32_t kGatherLag = 2;
constexpr int kNotListed = INT_MIN;   // slot past the entry's count

__device__ __forceinline__ bool run_producer_sparse(const Ctx& x, const Work& w,
                                                    const DecodeParams& prm,
                                                    const CUtensorMap* tm_q_rope, int lane,
                                                    int half) {
  const uint64_t gpolicy = ptx::policy_evict_first();
  SegIter it{w.b0, w.p0, w.b1, w.p1, w.items};
  int b, pb, pe;
  uint32_t g = 0, announced = 0, n_item = 0;
  const char* kv = static_cast<const char*>(prm.kv);
  const int32_t xq_rope = 512 + 32 * (int32_t)x.rank;
  const uint32_t lat_off = 512u * x.rank + 16u * (uint32_t)lane;
  const uint32_t rope_off = 1024u + 64u * x.rank + 16u * (uint32_t)(lane & 3);
  while (it.next(b, pb, pe)) {
    if (half == 0 && !wait_warp(x, x.bar(B_QEMPTY), (n_item & 1u) ^ 1u)) {
      ptx::cp_async_wait<0>();
      return false;
    }
    if (half == 0 && lane == 0) {
      ptx::mbar_arrive_expect_tx(x.bar(B_QFULL), kQRopeTx);
      const int32_t row0 = b * w.rows + w.tile * kTileRows;
      ptx::tma_load_2d(x.sbase + kQRope, tm_q_rope, xq_rope, row0, x.bar(B_QFULL));
    }
    const int count = prm.seqlens[b];
    const int cap = prm.cache_len[b];
    const int lim = count < prm.topk ? count : prm.topk;
    const int32_t* list = prm.indices + (size_t)b * prm.topk;
    const int32_t* bt = prm.block_table + (size_t)b * prm.max_pages;
    if (count > prm.topk && lane == 0 && half == 0) atomicCAS(x.err, 0, MLA_ERR_DEVICE_BOUNDS);
    // this lane's row of every chunk (lanes past kGatherRows repeat the first ones)
    const int myr = kGatherRows * half + (lane & (kGatherRows - 1));
    // list position of row r of chunk pg (kNotListed past the count)
    auto position = [&](int pg, int r) -> int {
      const int j = pg * kPageTokens + r;
      return (pg < pe && j < lim) ? list[j] : kNotListed;
    };
    // block-table entry of a position (the load is only issued here; the
    // value is looked at by `resolve`, a chunk later)
    auto page_of = [&](int t) -> int {
      return (t != kNotListed && t >= 0 && t < cap && t / kPageTokens < prm.max_pages)
                 ? bt[t / kPageTokens]
                 : -1;
    };
    // cache row (page * 64 + slot) of a position; -1 reads zeros
    auto resolve = [&](int t, int page) -> int {
      if (t == kNotListed) return -1;
      if ((unsigned)page >= (unsigned)prm.num_pages) {
        atomicCAS(x.err, 0, MLA_ERR_DEVICE_BOUNDS);
        return -1;
      }
      return page * kPageTokens + t % kPageTokens;
    };
    int t_cur = position(pb, myr);
    int p_cur = page_of(t_cur);
    int t_next = position(pb + 1, myr);
    for (int pg = pb; pg < pe; ++pg, ++g) {
      const int row = resolve(t_cur, p_cur);
      // one chunk ahead: the block-table entries of pg + 1; two ahead: the
      // positions of pg + 2
      t_cur = t_next;
      p_cur = page_of(t_cur);
      t_next = position(pg + 2, myr);
      const uint32_t s = g % kStages, k = g / kStages;
      if (!wait_warp(x, x.bar(B_EMPTY + s), (k & 1u) ^ 1u)) {
        ptx::cp_async_wait<0>();
        return false;
      }
      const uint32_t st = x.sbase + kStage0 + s * kStageBytes;
      const uint32_t box = st + (uint32_t)(lane >> 3) * 8192u;
#pragma unroll 4
      for (int r = kGatherRows * half; r < kGatherRows * (half + 1); ++r) {
        const int rr = __shfl_sync(0xffffffffu, row, r & (kGatherRows - 1));
        const uint32_t dst = box + (uint32_t)r * 128u + ((((uint32_t)lane & 7u) ^ ((uint32_t)r & 7u)) << 4);
        if (rr >= 0)
          ptx::cp_async16_full_hint(dst, kv + (size_t)rr * (kDqk * 2) + lat_off, gpolicy);
        else
          ptx::cp_async16(dst, kv, 0u);
      }
#pragma unroll
      for (int i = 0; i < kGatherRows / 8; ++i) {
        const int r = kGatherRows * half + 8 * i + (lane >> 2);
        const int rr = __shfl_sync(0xffffffffu, row, r & (kGatherRows - 1));
        const uint32_t dst = st + kStageRope + (uint32_t)r * 64u +
                             ((((uint32_t)lane & 3u) ^ (((uint32_t)r >> 1) & 3u)) << 4);
        if (rr >= 0)
          ptx::cp_async16_full_hint(dst, kv + (size_t)rr * (kDqk * 2) + rope_off, gpolicy);
        else
          ptx::cp_async16(dst, kv, 0u);
      }
      ptx::cp_async_commit();
      if (g >= announced + kGatherLag) {
        ptx::cp_async_wait<kGatherLag>();
        ptx::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(x.bar(B_FULL + announced % kStages));
        ++announced;
      }
    }
    ptx::cp_async_wait<0>();
    ptx::fence_proxy_async_smem();
    __syncwarp();
    for (; announced < g; ++announced)
      if (lane == 0) ptx::mbar_arrive(x.bar(B_FULL + announced % kStages));
    ++n_item;
  }
  return true;
}

// ------------------------------------------------------------------ MMA issuer
// Issues S = Q K^T for page gq and O += P V for page gp (gp < gq), each as
// soon as its inputs are ready, in page order within each kind.
__device__ __forceinline__ void issue_qk(const Ctx& x, uint32_t g) {
  constexpr uint32_t id_qk = ptx::idesc_bf16_f32(128, 64, 0, 0);
  const uint32_t st = x.sbase + kStage0 + (g % kStages) * kStageBytes;
  const uint32_t d_s = x.tmem + kColS + (g & 1u) * 64;
  // latent dims: A = Q from TMEM (8 columns = 16 dims per K-step), B = K page
#pragma unroll
  for (int k = 0; k < 16; ++k) {
    const uint64_t bdesc =
        ptx::smem_desc(st + (k >> 2) * 8192 + (k & 3) * 32, 16, 1024, ptx::kLayoutSw128);
    ptx::mma_ts_elect(d_s, x.tmem + kColQ + k * 8, bdesc, id_qk, k ? 1u : 0u);
  }
  // rotary dims: both operands from shared memory
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const uint64_t adesc = ptx::smem_desc(x.sbase + kQRope + k * 32, 16, 512, ptx::kLayoutSw64);
    const uint64_t bdesc = ptx::smem_desc(st + kStageRope + k * 32, 16, 512, ptx::kLayoutSw64);
    ptx::mma_ss_elect(d_s, adesc, bdesc, id_qk, 1u);
  }
}

__device__ __forceinline__ void issue_pv(const Ctx& x, uint32_t g, bool first) {
  constexpr uint32_t id_pv = ptx::idesc_bf16_f32(128, 256, 0, 1);
  const uint32_t vbase = x.sbase + kStage0 + (g % kStages) * kStageBytes;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    // V as the MN-major B operand: 64-dim swizzle atoms 8 KB apart along N,
    // 8-token row groups 1 KB apart along K; 16 tokens per K-step.
    const uint64_t bdesc = ptx::smem_desc(vbase + k * 2048, 8192, 1024, ptx::kLayoutSw128);
    const uint64_t adesc = ptx::smem_desc(x.sbase + kP + (g % kPBufs) * kPBytes + k * 32, 16, 1024,
                                          ptx::kLayoutSw128);
    ptx::mma_ss_elect(x.tmem + kColO, adesc, bdesc, id_pv, (first && k == 0) ? 0u : 1u);
  }
}

// Score MMAs, page by page, as soon as the page is loaded, the Q tile is in
// place and the page's TMEM score tile is free.
__device__ __forceinline__ bool run_mma_qk(const Ctx& x, const Work& w) {
  SegIter it{w.b0, w.p0, w.b1, w.p1, w.items};
  int b, pb, pe;
  uint32_t g = 0, n_item = 0;
  while (it.next(b, pb, pe)) {
    if (!wait_warp(x, x.bar(B_QFULL), n_item & 1u)) return false;
    for (int pg = pb; pg < pe; ++pg, ++g) {
      if (!wait_warp(x, x.bar(B_FULL + g % kStages), (g / kStages) & 1u)) return false;
      if (!wait_warp(x, x.bar(B_SEMPTY + (g & 1u)), ((g >> 1) & 1u) ^ 1u)) return false;
      ptx::tc_fence_after();
      issue_qk(x, g);
      ptx::mma_commit_elect(x.bar(B_SFULL + (g & 1u)));
    }
    ptx::mma_commit_elect(x.bar(B_QEMPTY));
    ++n_item;
  }
  return true;
}

// P.V MMAs, page by page, once the page's probabilities (all 128 rows) are
// in shared memory; the first page of a tile also waits until the previous
// tile's output has been read out of TMEM.
__device__ __forceinline__ bool run_mma_pv(const Ctx& x, const Work& w) {
  SegIter it{w.b0, w.p0, w.b1, w.p1, w.items};
  int b, pb, pe;
  uint32_t g = 0, n_item = 0;
  while (it.next(b, pb, pe)) {
    if (!wait_warp(x, x.bar(B_OEMPTY), (n_item & 1u) ^ 1u)) return false;
    for (int pg = pb; pg < pe; ++pg, ++g) {
      if (!wait_warp(x, x.bar(B_PFULL + g % kPBufs), (g / kPBufs) & 1u)) return false;
      ptx::tc_fence_after();
      issue_pv(x, g, pg == pb);
      ptx::mma_commit_elect(x.bar(B_EMPTY + g % kStages));
      ptx::mma_commit_elect(x.bar(B_PEMPTY + g % kPBufs));
    }
    ptx::mma_commit_elect(x.bar(B_OFULL));
    ++n_item;
  }
  return true;
}

// ------------------------------------------------------------------ half-quadrant TMEM access
// 16 lanes of one lane quadrant, two threads per lane: thread t reaches lane
// base + (t & 15) at columns col + (t >> 4) * OFF + j, j < 32 (the tcgen05
// .16x32bx2 shape; its layout was checked on GB300 against the 32x32b one).
// The load waits for its data in the same statement, as tmem_load32.
#define MLA_R32(i) "=r"(r[i])
template <int OFF>
__device__ __forceinline__ void tmem_load16x2(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.16x32bx2.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32], "
      "%33;\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : MLA_R32(0), MLA_R32(1), MLA_R32(2), MLA_R32(3), MLA_R32(4), MLA_R32(5), MLA_R32(6),
        MLA_R32(7), MLA_R32(8), MLA_R32(9), MLA_R32(10), MLA_R32(11), MLA_R32(12), MLA_R32(13),
        MLA_R32(14), MLA_R32(15), MLA_R32(16), MLA_R32(17), MLA_R32(18), MLA_R32(19),
        MLA_R32(20), MLA_R32(21), MLA_R32(22), MLA_R32(23), MLA_R32(24), MLA_R32(25),
        MLA_R32(26), MLA_R32(27), MLA_R32(28), MLA_R32(29), MLA_R32(30), MLA_R32(31)
      : "r"(taddr), "n"(OFF)
      : "memory");
}
#undef MLA_R32
#define MLA_W32(i) "r"(v[i])
template <int OFF>
__device__ __forceinline__ void tmem_store16x2(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.16x32bx2.x32.b32 [%0], %1, "
      "{%2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, "
      "%18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32, %33};" ::"r"(
          taddr),
      "n"(OFF), MLA_W32(0), MLA_W32(1), MLA_W32(2), MLA_W32(3), MLA_W32(4), MLA_W32(5),
      MLA_W32(6), MLA_W32(7), MLA_W32(8), MLA_W32(9), MLA_W32(10), MLA_W32(11), MLA_W32(12),
      MLA_W32(13), MLA_W32(14), MLA_W32(15), MLA_W32(16), MLA_W32(17), MLA_W32(18), MLA_W32(19),
      MLA_W32(20), MLA_W32(21), MLA_W32(22), MLA_W32(23), MLA_W32(24), MLA_W32(25), MLA_W32(26),
      MLA_W32(27), MLA_W32(28), MLA_W32(29), MLA_W32(30), MLA_W32(31)
      : "memory");
}
#undef MLA_W32

// This CTA's O columns of the 16 rows at `lanes` (a half quadrant) times each
// row's alpha (the two threads of a row hold the same alpha): 4 x 32 columns
// per thread, the 256 in all.
__device__ __forceinline__ void scale_o_rows(const Ctx& x, uint32_t lanes, float alpha) {
#pragma unroll 1
  for (int ch = 0; ch < 4; ++ch) {
    uint32_t v[32];
    const uint32_t ta = x.tmem + lanes + kColO + ch * 32;
    tmem_load16x2<128>(ta, v);
#pragma unroll
    for (int k = 0; k < 32; ++k) v[k] = __float_as_uint(__uint_as_float(v[k]) * alpha);
    tmem_store16x2<128>(ta, v);
  }
  ptx::tmem_wait_st();
}

// ------------------------------------------------------------------ page workers
// Warps 0-3 (set 0) take the even pages of the CTA's work, warps 4-7 (set 1)
// the odd ones; warp q of a set works on TMEM lane quadrant q, whose 32 rows
// are 16 of this CTA's (lanes 32 q + 16 r + [0, 16) in CTA r) and 16 of the
// peer's.  For its page, a worker
//  A. copies the score tile's partial scores out of TMEM (which frees it for
//     the page after next) and ships the peer's 16 rows with st.async into
//     the peer's receive buffer, as [16-byte chunk][owned row];
//  B. adds the peer's partial for its own 16 rows, two threads per row with
//     32 of the page's 64 columns each, masks, and takes the row max (the
//     accum_s -> scores_max reduce: over the thread's 32 columns, then with
//     its partner's);
//  C. takes the running max from the worker of the previous page (shared
//     memory and an mbarrier per quadrant), decides the rescale, and hands
//     the new running max on, so the online softmax stays sequential while
//     the rest of two consecutive pages overlaps;
//  D. writes the bf16 probabilities and rescale factors into P buffer g % 2
//     and bulk-copies them into the same places in the peer (once the peer's
//     buffer is free);
//  E. imports the peer's probabilities for its peer rows (rescaling those rows
//     of O when a factor is not 1) and signals the P.V issuer.
// Each worker keeps the probability sums of its own pages, scaled to the
// running max it last saw; at the end of a tile set 1 hands its sums to set
// 0, which finishes the tile: O / l for all 32 rows of its quadrant and this
// CTA's half of the output dims, and lse for its own rows.  Set 1 also puts
// the latent half of each Q tile into TMEM (one row per thread).
__device__ __forceinline__ bool run_pages(const Ctx& x, const Work& w, const DecodeParams& prm,
                                          int set, int quad, int lane) {
  const int half = lane >> 4;
  const int t = lane & 15;
  const int ro = quad * 32 + kSubRows * (int)x.rank + t;   // owned tile row (TMEM lane)
  const int hr = kSubRows * quad + t;                      // its owned-row index
  const uint32_t own_lanes = (uint32_t)(quad * 32 + kSubRows * (int)x.rank) << 16;
  const uint32_t peer_lanes = (uint32_t)(quad * 32 + kSubRows * (int)x.peer) << 16;
  const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
  const uint32_t chunk0 = (uint32_t)(6 * half) * (kHalfRows * 16);
  const uint32_t recv_row = x.sbase + kRecv + (uint32_t)hr * 16u + chunk0;
  const uint32_t peer_row = ptx::map_to_rank(x.sbase + kRecv, x.peer) + (uint32_t)hr * 16u + chunk0;
  const uint32_t peer_rfull = ptx::map_to_rank(x.bar(B_RFULL), x.peer);
  const uint32_t peer_rempty = ptx::map_to_rank(x.bar(B_REMPTY), x.peer);
  const uint32_t peer_precv = ptx::map_to_rank(x.bar(B_PRECV), x.peer);
  const uint32_t peer_lrecv = ptx::map_to_rank(x.bar(B_LRECV), x.peer);
  const uint32_t peer_base = ptx::map_to_rank(x.sbase, x.peer);
  const uint32_t alpha_in = x.sbase + kAlpha + (x.peer * kHalfRows + (uint32_t)hr) * 4u;
  const uint32_t hand_out = x.sbase + kHand + ((uint32_t)(set * 4 + quad) * kSubRows + t) * 4u;
  const uint32_t hand_in = x.sbase + kHand + ((uint32_t)((set ^ 1) * 4 + quad) * kSubRows + t) * 4u;
  const uint32_t pswz = (uint32_t)(ro & 7);
  const float scale_log2 = prm.scale_log2;
  const __nv_bfloat16* q = static_cast<const __nv_bfloat16*>(prm.q);

  SegIter it{w.b0, w.p0, w.b1, w.p1, w.items};
  int b, pb, pe;
  uint32_t g = 0, n_item = 0;
  while (it.next(b, pb, pe)) {
    if (set == 1) {
      // Q latent half of this tile -> TMEM columns [kColQ, kColQ + 128) once
      // the previous tile's last score MMA is done.  Rows past the batch
      // entry's query rows are zero.  All 32 loads of the row are issued
      // before the first use: the tile's first score MMA waits on this.
      if (!wait_warp(x, x.bar(B_QEMPTY), (n_item & 1u) ^ 1u)) return false;
      const int qr = w.tile * kTileRows + quad * 32 + lane;
      const bool valid = qr < w.rows;
      const uint4* src = reinterpret_cast<const uint4*>(
          q + ((int64_t)b * w.rows + (valid ? qr : 0)) * kDqk + 256 * (int)x.rank);
      uint4 qv[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) qv[j] = valid ? src[j] : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
      for (int ch = 0; ch < 4; ++ch) {
        uint32_t v[32];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          v[4 * j] = qv[ch * 8 + j].x;
          v[4 * j + 1] = qv[ch * 8 + j].y;
          v[4 * j + 2] = qv[ch * 8 + j].z;
          v[4 * j + 3] = qv[ch * 8 + j].w;
        }
        ptx::tmem_st32(x.tmem + lane_base + kColQ + ch * 32, v);
      }
      ptx::tmem_wait_st();
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(x.bar(B_QFULL));
    }

    const int qo = w.tile * kTileRows + ro;
    const bool valid_o = qo < w.rows;
    const int io = qo / prm.h_q;
    const int ho = qo - io * prm.h_q;
    const int L = prm.seqlens[b];
    const int n_valid = valid_o ? L - prm.s_q + 1 + io : 0;
    const int P_total = w.items[b * kItemWords + 0];
    // m_run: the running max this worker's sums are scaled to.  l_run sums
    // the fp32 probabilities (for lse); lb_run sums them after the bf16
    // rounding the P.V MMA sees, so out = sum(p v) / sum(p) uses one set of
    // weights and stays a true weighted average of the value rows.  Each
    // thread sums its 32 columns of this worker's pages.
    float m_run = -INFINITY, l_run = 0.f, lb_run = 0.f;

    for (int pg = pb; pg < pe; ++pg, ++g) {
      if ((int)(g & 1u) != set) continue;
      const bool first = (pg == pb);
      const uint32_t sb = g & 1u;             // score tile
      const uint32_t rb = g % kRBufs;         // receive buffer
      const uint32_t pbuf = g % kPBufs;       // P buffer

      // A. Partial scores out of TMEM; the peer's rows to the peer.
      if (quad == 0 && lane == 0) ptx::mbar_arrive_expect_tx(x.bar(B_RFULL + rb), kRecvBytes);
      if (!wait_warp(x, x.bar(B_SFULL + sb), (g >> 1) & 1u)) return false;
      ptx::tc_fence_after();
      uint32_t v[32];
      float s[32];
      tmem_load16x2<32>(x.tmem + peer_lanes + kColS + sb * 64, v);
      {
        uint32_t u[32];
        tmem_load16x2<32>(x.tmem + own_lanes + kColS + sb * 64, u);
#pragma unroll
        for (int k = 0; k < 32; ++k) s[k] = __uint_as_float(u[k]);
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(x.bar(B_SEMPTY + sb));
      // the peer has read what was sent into this buffer kRBufs pages ago
      if (!wait_warp(x, x.bar(B_REMPTY + rb), ((g / kRBufs) & 1u) ^ 1u, true)) return false;
      // 24-bit floats: the rounding (<= 2^-16 relative) is within what the
      // fp32 accumulation of these 288 products already allows (288 x 2^-24
      // of the sum of their magnitudes), and the transfer, which bounds the
      // page rate, shrinks by a quarter
      uint32_t w24[24];
#pragma unroll
      for (int j = 0; j < 8; ++j)
        ptx::pack24x4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3], w24[3 * j],
                      w24[3 * j + 1], w24[3 * j + 2]);
#pragma unroll
      for (int c = 0; c < 6; ++c)
        ptx::st_async_v4_b32(peer_row + rb * kRecvBytes + (uint32_t)c * (kHalfRows * 16),
                             w24[4 * c], w24[4 * c + 1], w24[4 * c + 2], w24[4 * c + 3],
                             peer_rfull + 8u * rb);

      // B. Full scores of my rows, mask, row max.
      if (!wait_warp(x, x.bar(B_RFULL + rb), (g / kRBufs) & 1u, true)) return false;
      {
        uint32_t w24[24];
#pragma unroll
        for (int c = 0; c < 6; ++c) {
          const uint4 r4 = ptx::ld_shared_v4u(recv_row + rb * kRecvBytes + (uint32_t)c * (kHalfRows * 16));
          w24[4 * c] = r4.x;
          w24[4 * c + 1] = r4.y;
          w24[4 * c + 2] = r4.z;
          w24[4 * c + 3] = r4.w;
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          float a, bq, c2, d;
          ptx::unpack24x4(w24[3 * j], w24[3 * j + 1], w24[3 * j + 2], a, bq, c2, d);
          ptx::f2_unpack(ptx::f2_add(ptx::f2_pack(s[4 * j], s[4 * j + 1]), ptx::f2_pack(a, bq)),
                         s[4 * j], s[4 * j + 1]);
          ptx::f2_unpack(ptx::f2_add(ptx::f2_pack(s[4 * j + 2], s[4 * j + 3]), ptx::f2_pack(c2, d)),
                         s[4 * j + 2], s[4 * j + 3]);
        }
      }
      const int tok0 = pg * kPageTokens + 32 * half;
      if (__any_sync(0xffffffffu, tok0 + 32 > n_valid)) {
#pragma unroll
        for (int k = 0; k < 32; ++k)
          if (tok0 + k >= n_valid) s[k] = -INFINITY;
      }
      float m4[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float* sj = s + 8 * j;
        m4[j] = fmaxf(ptx::max3(ptx::max3(ptx::max3(sj[0], sj[1], sj[2]), sj[3], sj[4]), sj[5], sj[6]),
                      sj[7]);
      }
      float mx = fmaxf(ptx::max3(m4[0], m4[1], m4[2]), m4[3]);
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
      // Every value read from the receive buffer went into mx: once mx is
      // computed the reads are complete and the peer may refill the buffer.
      ptx::consume(mx);
      __syncwarp();
      if (lane == kRemoteLane) ptx::mbar_arrive_cluster_relaxed(peer_rempty + 8u * rb);

      // C. Running max: from the previous page's worker, to the next one's.
      float m_ref = -INFINITY;
      if (g > 0) {
        if (!wait_warp(x, x.bar(B_HAND + (uint32_t)((set ^ 1) * 4 + quad)), ((g - 1) >> 1) & 1u))
          return false;
        if (!first) m_ref = __uint_as_float(ptx::ld_shared_u32_volatile(hand_in));
      }
      const float m_cand = fmaxf(m_ref, mx * scale_log2);   // scale_log2 > 0
      const bool rescale = !first && (m_cand > m_ref + kRescaleThreshold);
      const float m_new = (first || rescale) ? m_cand : m_ref;
      const float alpha = rescale ? ptx::ex2(m_ref - m_new) : 1.0f;   // O's factor
      if (m_new != m_run) {
        // this worker's sums were taken at an older running max
        const float f = (m_run == -INFINITY) ? 0.f : ptx::ex2(m_run - m_new);
        l_run *= f;
        lb_run *= f;
        m_run = m_new;
      }
      if (half == 0) ptx::st_shared_u32(hand_out, __float_as_uint(m_new));
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(x.bar(B_HAND + (uint32_t)(set * 4 + quad)));

      const float neg_m = (m_new == -INFINITY) ? 0.f : -m_new;
      // exp2(s * scale - m) on pairs: the fma and the sums are f32x2 ops, and
      // the sums run as two independent chains
      uint32_t pk[16];
      const uint64_t sc2 = ptx::f2_pack(scale_log2, scale_log2);
      const uint64_t nm2 = ptx::f2_pack(neg_m, neg_m);
      uint64_t ps2[2] = {0ull, 0ull}, pb2[2] = {0ull, 0ull};
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        float xa, xc;
        ptx::f2_unpack(ptx::f2_fma(ptx::f2_pack(s[2 * j], s[2 * j + 1]), sc2, nm2), xa, xc);
        const float a = ptx::ex2(xa), c = ptx::ex2(xc);
        ps2[j & 1] = ptx::f2_add(ps2[j & 1], ptx::f2_pack(a, c));
        pk[j] = ptx::pack_bf16x2(a, c);
        pb2[j & 1] = ptx::f2_add(pb2[j & 1], ptx::f2_pack(__uint_as_float(pk[j] << 16),
                                                          __uint_as_float(pk[j] & 0xffff0000u)));
      }
      float pa, pc, ba, bc;
      ptx::f2_unpack(ptx::f2_add(ps2[0], ps2[1]), pa, pc);
      ptx::f2_unpack(ptx::f2_add(pb2[0], pb2[1]), ba, bc);
      l_run += pa + pc;
      lb_run += ba + bc;

      // D. P buffer g % 2 is free: my P.V of page g - 2 is done and this
      //    warp's copy of page g - 2 to the peer has read its rows.  A
      //    rescale of O also needs the P.V of page g - 1 done.
      if (!wait_warp(x, x.bar(B_PEMPTY + pbuf), ((g / kPBufs) & 1u) ^ 1u)) return false;
      if (lane == kRemoteLane) ptx::bulk_wait_read_all();
      __syncwarp();
      if (__any_sync(0xffffffffu, rescale)) {
        if (kPBufs > 1 &&
            !wait_warp(x, x.bar(B_PEMPTY + (g - 1) % kPBufs), ((g - 1) / kPBufs) & 1u))
          return false;
        ptx::tc_fence_after();
        scale_o_rows(x, own_lanes, alpha);
      }
      // Past the end of the sequence the cache slots of the last page hold
      // stale data; their probabilities are exactly 0 but 0 * NaN is NaN in
      // the P.V MMA, so zero those value rows first (each CTA zeroes its own
      // stage, split between the page's four workers).
      if (pg == P_total - 1 && (L & (kPageTokens - 1)) != 0) {
        const int t0 = L & (kPageTokens - 1);
        const uint32_t st = x.sbase + kStage0 + (g % kStages) * kStageBytes;
        const int n16 = (kPageTokens - t0) * 4 * 8;   // 16-byte pieces: rows x 4 boxes x 8
        for (int idx = quad * 32 + lane; idx < n16; idx += 4 * 32) {
          const int row = t0 + (idx >> 5), box = (idx >> 3) & 3, c16 = idx & 7;
          ptx::st_shared_v4(st + box * 8192 + row * 128 + c16 * 16, 0u, 0u, 0u, 0u);
        }
      }
      {
        // P row ro, 128-byte swizzle: 16-byte chunk c at position c ^ (ro % 8);
        // this thread's 32 columns are chunks 4 half .. 4 half + 3
        const uint32_t prow = x.sbase + kP + pbuf * kPBytes + (uint32_t)ro * 128u;
#pragma unroll
        for (int j = 0; j < 4; ++j)
          ptx::st_shared_v4(prow + (((uint32_t)(4 * half + j) ^ pswz) << 4), pk[4 * j],
                            pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
        if (half == 0)
          ptx::st_shared_u32(x.sbase + kAlpha + pbuf * kAlphaBufBytes +
                                 (x.rank * kHalfRows + (uint32_t)hr) * 4u,
                             __float_as_uint(alpha));
      }
      ptx::fence_proxy_async_smem();
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(x.bar(B_PFULL + pbuf));
      // this warp's 16 P rows (2 KB, contiguous in the swizzled buffer) and
      // their factors into the peer once its buffer is free; they complete on
      // the peer's PRECV barrier
      if (!wait_warp(x, x.bar(B_PFREE + pbuf), (g / kPBufs) & 1u, true)) return false;
      if (lane == kRemoteLane) {
        const uint32_t poff = kP + pbuf * kPBytes + (uint32_t)(quad * 32 + kSubRows * (int)x.rank) * 128u;
        const uint32_t aoff = kAlpha + pbuf * kAlphaBufBytes + (x.rank * kHalfRows + kSubRows * quad) * 4u;
        ptx::bulk_copy_to_peer(peer_base + poff, x.sbase + poff, kSubRows * 128u, peer_precv + 8u * pbuf);
        ptx::bulk_copy_to_peer(peer_base + aoff, x.sbase + aoff, kSubRows * 4u, peer_precv + 8u * pbuf);
        ptx::bulk_commit();
      }

      // E. The peer's rows of this page.
      if (!wait_warp(x, x.bar(B_PRECV + pbuf), (g / kPBufs) & 1u, true)) return false;
      const float alpha_p =
          __uint_as_float(ptx::ld_shared_u32_volatile(alpha_in + pbuf * kAlphaBufBytes));
      if (__any_sync(0xffffffffu, alpha_p != 1.0f)) {
        if (kPBufs > 1 &&
            !wait_warp(x, x.bar(B_PEMPTY + (g - 1) % kPBufs), ((g - 1) / kPBufs) & 1u))
          return false;
        ptx::tc_fence_after();
        scale_o_rows(x, peer_lanes, alpha_p);
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(x.bar(B_PFULL + pbuf));
    }

    // End of the tile.
    const uint32_t par = n_item & 1u;
    const uint32_t sums = x.sbase + kSums + ((par * 4 + (uint32_t)quad) * 32 + (uint32_t)lane) * 12u;
    const int ns = w.items[b * kItemWords + 1];
    const bool direct = (ns == 1);
    const int sidx = (n_item == 0) ? w.split0 : 0;
    const int64_t slot = (int64_t)w.tile * w.stotal + w.items[b * kItemWords + 2] + sidx;
    // rows of the epilogue: lane -> tile row quad * 32 + lane (mine when its
    // half quadrant is this CTA's, and then this thread owned it)
    const int re = quad * 32 + lane;
    const int qe = w.tile * kTileRows + re;
    const bool valid_e = qe < w.rows;
    const int ie = qe / prm.h_q;
    const int he = qe - ie * prm.h_q;
    const int64_t orow = ((int64_t)b * prm.s_q + ie) * prm.h_q + he;
    // O / l for this CTA's columns [32 ch0, 32 ch1) of the row, to the final
    // output or to this split's partial slot
    auto drain = [&](int ch0, int ch1, float inv_l) {
      ptx::tc_fence_after();
#pragma unroll 1
      for (int ch = ch0; ch < ch1; ++ch) {
        uint32_t o[32];
        tmem_load32(x.tmem + lane_base + kColO + ch * 32, o);
        if (valid_e) {
          const int d0 = (int)x.rank * 256 + ch * 32;
          if (direct && !prm.out_f32) {
            // a row's 32 dims: 64 bytes, rows 1 KB apart (32-byte stores
            // when out allows: whole sectors)
            uint32_t pk[16];
#pragma unroll
            for (int k = 0; k < 16; ++k)
              pk[k] = ptx::pack_bf16x2(__uint_as_float(o[2 * k]) * inv_l,
                                       __uint_as_float(o[2 * k + 1]) * inv_l);
            __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(prm.out) + orow * kDv + d0;
            if (prm.out_v8) {
              ptx::st_global_v8(dst, pk[0], pk[1], pk[2], pk[3], pk[4], pk[5], pk[6], pk[7]);
              ptx::st_global_v8(dst + 16, pk[8], pk[9], pk[10], pk[11], pk[12], pk[13], pk[14], pk[15]);
            } else {
#pragma unroll
              for (int qq = 0; qq < 4; ++qq)
                reinterpret_cast<uint4*>(dst)[qq] =
                    make_uint4(pk[4 * qq], pk[4 * qq + 1], pk[4 * qq + 2], pk[4 * qq + 3]);
            }
          } else {
            // fp32: the final output row (fp32 out), or this split's partial
            // ([dim / 4][row][4] in the workspace slot)
            float4* base = direct ? reinterpret_cast<float4*>(static_cast<float*>(prm.out) +
                                                              orow * kDv + d0)
                                  : reinterpret_cast<float4*>(prm.ws_o) +
                                        slot * (kDv / 4) * kTileRows +
                                        (int64_t)(d0 / 4) * kTileRows + re;
            const int64_t step = direct ? 1 : kTileRows;
#pragma unroll
            for (int qq = 0; qq < 8; ++qq)
              base[qq * step] = make_float4(__uint_as_float(o[4 * qq]) * inv_l,
                                            __uint_as_float(o[4 * qq + 1]) * inv_l,
                                            __uint_as_float(o[4 * qq + 2]) * inv_l,
                                            __uint_as_float(o[4 * qq + 3]) * inv_l);
          }
        }
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(x.bar(B_OEMPTY));
    };
    if (set == 1) {
      // hand this worker's sums (and the max they are scaled to) to set 0,
      // once set 0 has read those of the tile before last; then drain the
      // upper half of this CTA's columns once set 0 has published 1/l
      if (!wait_warp(x, x.bar(B_SUMSFREE + par), ((n_item >> 1) & 1u) ^ 1u)) return false;
      ptx::st_shared_u32(sums, __float_as_uint(m_run));
      ptx::st_shared_u32(sums + 4, __float_as_uint(l_run));
      ptx::st_shared_u32(sums + 8, __float_as_uint(lb_run));
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(x.bar(B_SUMS + par));
      if (!wait_warp(x, x.bar(B_EPI), n_item & 1u)) return false;
      if (!wait_warp(x, x.bar(B_OFULL), n_item & 1u)) return false;
      drain(4, 8, __uint_as_float(ptx::ld_shared_u32_volatile(x.sbase + kEpiInv + (uint32_t)re * 4u)));
      ++n_item;
      continue;
    }
    if (!wait_warp(x, x.bar(B_SUMS + par), (n_item >> 1) & 1u)) return false;
    {
      const float m1 = __uint_as_float(ptx::ld_shared_u32_volatile(sums));
      const float l1 = __uint_as_float(ptx::ld_shared_u32_volatile(sums + 4));
      const float lb1 = __uint_as_float(ptx::ld_shared_u32_volatile(sums + 8));
      const float m = fmaxf(m_run, m1);
      const float f0 = (m_run == -INFINITY) ? 0.f : ptx::ex2(m_run - m);
      const float f1 = (m1 == -INFINITY) ? 0.f : ptx::ex2(m1 - m);
      l_run = l_run * f0 + l1 * f1;
      lb_run = lb_run * f0 + lb1 * f1;
      m_run = m;
    }
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive(x.bar(B_SUMSFREE + par));
    // Epilogue: O / l for this CTA's dims of the warp's 32 rows; lse by the
    // row's owner.  The owners' sums are final after the last page: they send
    // 1/l of their rows to the peer and write lse before the last P.V is
    // done, so that draining O (which the next tile's first P.V waits for) is
    // all that follows it.
    l_run += __shfl_xor_sync(0xffffffffu, l_run, 16);
    lb_run += __shfl_xor_sync(0xffffffffu, lb_run, 16);
    const float inv_own = lb_run > 0.f ? 1.0f / lb_run : 0.f;
    if (half == 0)
      ptx::st_shared_u32(x.sbase + kInvL + par * 512u + (x.rank * kHalfRows + (uint32_t)hr) * 4u,
                         __float_as_uint(inv_own));
    ptx::fence_proxy_async_smem();
    __syncwarp();
    if (lane == kRemoteLane) {
      // this warp's 16 values of 1/l
      const uint32_t woff = kInvL + par * 512u + (x.rank * kHalfRows + kSubRows * quad) * 4u;
      ptx::bulk_copy_to_peer(ptx::map_to_rank(x.sbase + woff, x.peer), x.sbase + woff,
                             kSubRows * 4u, peer_lrecv + 8u * par);
      ptx::bulk_commit();
      ptx::bulk_wait_read_all();
    }
    if (quad == 0 && lane == 0) ptx::mbar_arrive_expect_tx(x.bar(B_LRECV + par), kInvLTx);
    if (half == 0 && valid_o) {
      const float lse_v = l_run > 0.f ? (m_run + log2f(l_run)) * kLn2 : -INFINITY;
      if (direct)
        prm.lse[((int64_t)b * prm.h_q + ho) * prm.s_q + io] = lse_v;
      else
        prm.ws_lse[slot * kTileRows + ro] = lse_v;
    }
    if (!wait_warp(x, x.bar(B_OFULL), n_item & 1u)) return false;
    if (!wait_warp(x, x.bar(B_LRECV + par), (n_item >> 1) & 1u, true)) return false;
    const float inv_l =
        (half == (int)x.rank)
            ? inv_own
            : __uint_as_float(ptx::ld_shared_u32_volatile(
                  x.sbase + kInvL + par * 512u + (x.peer * kHalfRows + (uint32_t)hr) * 4u));
    // publish 1/l of row re for set 1 (set 1 reads it before it arrives on
    // OEMPTY, and the next tile's 1/l is written only after that tile's
    // first P.V, which waits for OEMPTY)
    ptx::st_shared_u32(x.sbase + kEpiInv + (uint32_t)re * 4u, __float_as_uint(inv_l));
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive(x.bar(B_EPI));
    drain(0, 4, inv_l);
    ++n_item;
  }
  return true;
}

// ------------------------------------------------------------------ P notifier
// One thread.  Per page g: once this CTA's P.V of page g - 2 is done, its P
// buffer g % 2 may take the peer's rows of page g: post their byte count on
// PRECV and tell the peer (whose page workers then copy their rows in).
__device__ __forceinline__ bool run_pnotify(const Ctx& x, const Work& w) {
  const uint32_t peer_pfree = ptx::map_to_rank(x.bar(B_PFREE), x.peer);
  SegIter it{w.b0, w.p0, w.b1, w.p1, w.items};
  int b, pb, pe;
  uint32_t g = 0;
  while (it.next(b, pb, pe)) {
    for (int pg = pb; pg < pe; ++pg, ++g) {
      const uint32_t sb = g % kPBufs, ph = (g / kPBufs) & 1u;
      if (!wait_bar(x, x.bar(B_PEMPTY + sb), ph ^ 1u)) return false;
      ptx::mbar_arrive_expect_tx_relaxed(x.bar(B_PRECV + sb), kPRecvTx);
      ptx::mbar_arrive_cluster_relaxed(peer_pfree + 8u * sb);
    }
  }
  return true;
}

// Two instantiations: dense (kDenseThreads, the register budget of 384
// threads) and sparse (kThreads, with the extra gather warps).
template <bool kSparse>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kSparse ? kThreads : kDenseThreads, 1)
    mla_decode_kernel(const __grid_constant__ CUtensorMap tm_q_rope,
                      const __grid_constant__ CUtensorMap tm_kv_lat,
                      const __grid_constant__ CUtensorMap tm_kv_rope, const DecodeParams prm) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = ptx::cluster_ctarank();
  const int cluster = (int)(blockIdx.x >> 1);

  Ctx x;
  x.sbase = (ptx::smem_addr(smem_raw) + 1023u) & ~1023u;
  x.rank = rank;
  x.peer = rank ^ 1u;
  x.err = prm.err;
  const uint32_t tmem_slot = x.sbase + kMisc;
  x.abort_addr = x.sbase + kMisc + 4;
  x.peer_abort_addr = ptx::map_to_rank(x.abort_addr, x.peer);

  // Set-up that needs nothing from earlier kernels; with programmatic
  // dependent launch it overlaps the planner's tail.
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(x.bar(B_FULL + s), kSparse ? kGatherWarps : 1);   // gather warps, or the TMA
      ptx::mbar_init(x.bar(B_EMPTY + s), 1);
    }
    ptx::mbar_init(x.bar(B_QFULL), 1 + 4);   // rotary TMA + set 1's 4 warps
    ptx::mbar_init(x.bar(B_QEMPTY), 1);
    for (int s = 0; s < 2; ++s) {
      ptx::mbar_init(x.bar(B_SFULL + s), 1);
      ptx::mbar_init(x.bar(B_SEMPTY + s), 4);   // the page's 4 workers
      ptx::mbar_init(x.bar(B_RFULL + s), 1);    // own expect_tx + the peer's st.async bytes
      ptx::mbar_init(x.bar(B_REMPTY + s), 4);   // the peer's 4 workers of the page (remote)
      ptx::mbar_init(x.bar(B_LRECV + s), 1);    // own expect_tx + the peer's 1/l bytes
      ptx::mbar_init(x.bar(B_PFULL + s), 8);    // the page's 4 workers: own rows, then imported rows
      ptx::mbar_init(x.bar(B_SUMS + s), kQuadWarps);
      ptx::mbar_init(x.bar(B_SUMSFREE + s), kQuadWarps);
      ptx::mbar_init(x.bar(B_PEMPTY + s), 1);
      ptx::mbar_init(x.bar(B_PRECV + s), 1);    // own expect_tx + the peer's P bytes
      ptx::mbar_init(x.bar(B_PFREE + s), 1);    // the peer's P notifier (remote)
    }
    ptx::mbar_init(x.bar(B_OFULL), 1);
    for (int h = 0; h < 8; ++h) ptx::mbar_init(x.bar(B_HAND + h), 1);
    ptx::mbar_init(x.bar(B_OEMPTY), 2 * kQuadWarps);
    ptx::mbar_init(x.bar(B_EPI), kQuadWarps);
    ptx::mbar_init(x.bar(B_TEARDOWN), 2);   // both MMA-issuing threads
    ptx::st_shared_u32(x.abort_addr, 0u);
    ptx::fence_mbarrier_init();
  }
  if (warp == kMmaWarp) {
    ptx::tmem_alloc(tmem_slot, kTmemCols);
    ptx::tmem_relinquish();
  }
  if (warp == kProducerWarp && lane == 0) {
    ptx::prefetch_tmap(&tm_q_rope);
    ptx::prefetch_tmap(&tm_kv_lat);
    ptx::prefetch_tmap(&tm_kv_rope);
  }
  ptx::tc_fence_before();
  ptx::cluster_sync();   // both CTAs' barriers initialised and TMEM allocated
  ptx::tc_fence_after();
  x.tmem = ptx::ld_shared_u32_volatile(tmem_slot);

  // The plan (and the inputs) come from earlier kernels on the stream.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  // The plan must describe this call.  Both CTAs of a cluster read the same
  // plan and take the same branch.
  const int32_t* plan = prm.plan;
  Work w;
  bool has_work = false;
  // The group size follows from the grid and the call's shape, so this
  // cluster's entry is read in the same memory round trip as the header
  // (it lies inside any plan of this call's shape, whose size the caller
  // must provide); the header then decides whether it is used.
  const int tiles_l = plan_tiles(prm.s_q, prm.h_q);
  const int gt_l = plan_group_clusters((int)(gridDim.x >> 1), tiles_l);
  const int tile_l = gt_l > 0 ? cluster / gt_l : tiles_l;
  const int c_l = gt_l > 0 ? cluster - tile_l * gt_l : 0;
  const int32_t* cl = plan + H_WORDS + c_l * kClusterWords;
  const int e_b0 = cl[0], e_p0 = cl[1], e_b1 = cl[2], e_p1 = cl[3], e_s0 = cl[4];
  if (plan[H_MAGIC] != kPlanMagic || plan[H_BATCH] != prm.batch || plan[H_SQ] != prm.s_q ||
      plan[H_HQ] != prm.h_q || plan[H_NCLUSTERS] != (int)(gridDim.x >> 1) ||
      plan[H_GT] != gt_l || plan[H_TILES] != tiles_l || gt_l <= 0) {
    if (threadIdx.x == 0 && rank == 0) atomicCAS(prm.err, 0, MLA_ERR_PLAN);
  } else {
    const int gused = plan[H_GUSED];
    w.tile = tile_l;
    if (w.tile < tiles_l && c_l < gused) {
      w.b0 = e_b0;
      w.p0 = e_p0;
      w.b1 = e_b1;
      w.p1 = e_p1;
      w.split0 = e_s0;
      if (w.b0 < 0 || w.p0 < 0 || w.p1 < 0 || w.b0 > w.b1 || w.b1 > prm.batch ||
          (w.b1 == prm.batch && w.p1 != 0)) {
        if (threadIdx.x == 0 && rank == 0) atomicCAS(prm.err, 0, MLA_ERR_PLAN);
      } else if (!(w.b0 == w.b1 && w.p0 >= w.p1)) {
        has_work = true;
        w.rows = prm.s_q * prm.h_q;
        w.stotal = plan[H_STOTAL];
        w.items = plan + plan_off_items(gt_l) / 4;
      }
    }
  }

  if (!has_work) {
    // nothing to do: fall through to the teardown
  } else if (warp == kProducerWarp || warp >= kGatherWarp) {
    if constexpr (kSparse)
      run_producer_sparse(x, w, prm, &tm_q_rope, lane,
                          warp == kProducerWarp ? 0 : warp - kGatherWarp + 1);
    else if (warp == kProducerWarp && lane == 0)
      run_producer(x, w, prm, &tm_q_rope, &tm_kv_lat, &tm_kv_rope);
    __syncwarp();
  } else if (warp == kMmaWarp) {
    run_mma_qk(x, w);   // whole warp: one elected lane issues
    __syncwarp();
  } else if (warp == kPvWarp) {
    run_mma_pv(x, w);
    __syncwarp();
  } else if (warp == kPSendWarp) {
    if (lane == 0) run_pnotify(x, w);
    __syncwarp();
  } else if (warp < 2 * kQuadWarps) {
    run_pages(x, w, prm, warp / kQuadWarps, warp % kQuadWarps, lane);
    __syncwarp();
  }

  // Teardown.  After an abort, give in-flight copies and MMAs time to land
  // before the shared memory and TMEM are released.
  const bool aborted = ptx::ld_shared_u32_volatile(x.abort_addr) != 0u;
  if (warp == kMmaWarp || warp == kPvWarp) {
    // each issuing lane's MMAs are done (the warp is converged here, so the
    // commit goes out from the lane that issued them)
    ptx::mma_commit_elect(x.bar(B_TEARDOWN));
    const uint64_t t0 = ptx::globaltimer();
    while (!ptx::mbar_try_wait(x.bar(B_TEARDOWN), 0u)) {
      if (ptx::globaltimer() - t0 > kWaitTimeoutNs) {
        if (lane == 0) atomicCAS(x.err, 0, MLA_ERR_DEVICE_TIMEOUT);
        break;
      }
    }
  }
  if (aborted) {
    const uint64_t t0 = ptx::globaltimer();
    while (ptx::globaltimer() - t0 < kDrainNs) __nanosleep(1000);
  }
  __syncwarp();
  ptx::tc_fence_before();
  ptx::cluster_sync();   // no remote traffic into either CTA after this point
  if (warp == kMmaWarp) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(x.tmem, kTmemCols);
  }
}

// Self-test of the failure path: a two-CTA cluster whose only wait, on an
// mbarrier nothing arrives on, goes through wait_bar.  The first CTA to give
// up (after kWaitTimeoutNs) records MLA_ERR_DEVICE_TIMEOUT and raises both
// CTAs' abort flags, the other sees its flag and gives up too, and both
// leave through a cluster barrier, as the decode kernel's teardown does.
__global__ void __cluster_dims__(2, 1, 1) mla_wait_selftest_kernel(int* err) {
  __shared__ __align__(8) uint64_t never;
  __shared__ uint32_t abort_flag;
  const uint32_t rank = ptx::cluster_ctarank();
  Ctx x = {};
  x.rank = rank;
  x.peer = rank ^ 1u;
  x.abort_addr = ptx::smem_addr(&abort_flag);
  x.peer_abort_addr = ptx::map_to_rank(x.abort_addr, x.peer);
  x.err = err;
  const uint32_t bar = ptx::smem_addr(&never);
  if (threadIdx.x == 0) {
    ptx::mbar_init(bar, 1);
    ptx::st_shared_u32(x.abort_addr, 0u);
    ptx::fence_mbarrier_init();
  }
  ptx::cluster_sync();
  if (threadIdx.x == 0) wait_bar(x, bar, 0u);
  __syncwarp();
  ptx::cluster_sync();   // no remote store into either CTA after this point
}

}  // namespace

cudaError_t launch_wait_selftest(int* err, cudaStream_t stream) {
  mla_wait_selftest_kernel<<<2, 32, 0, stream>>>(err);
  return cudaGetLastError();
}

int decode_smem_bytes() { return (int)kSmemAlloc; }

cudaError_t decode_kernel_setup(int /*device*/) {
  const cudaError_t e = cudaFuncSetAttribute(
      mla_decode_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemAlloc);
  if (e != cudaSuccess) return e;
  const cudaError_t e2 = cudaFuncSetAttribute(
      mla_decode_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemAlloc);
  if (e2 != cudaSuccess) return e2;
  return narrow_kernel_setup();
}

int decode_max_clusters(int device) {
  int prev = 0;
  if (cudaGetDevice(&prev) != cudaSuccess) return -1;
  if (prev != device && cudaSetDevice(device) != cudaSuccess) return -1;
  int n = -1;
  if (decode_kernel_setup(device) == cudaSuccess) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * 1024, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = (size_t)kSmemAlloc;
    int m = 0;
    // the sparse instantiation (more threads) bounds both; the narrow
    // kernel runs on the same plans, so it bounds the count too
    if (cudaOccupancyMaxActiveClusters(&m, mla_decode_kernel<true>, &cfg) == cudaSuccess) n = m;
    const int mn = narrow_max_clusters();
    if (n > 0 && (mn < 0 || mn < n)) n = mn;
  }
  if (prev != device) cudaSetDevice(prev);
  return n;
}

cudaError_t launch_decode(const TensorMaps& m, const DecodeParams& p, int num_clusters,
                          cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * num_clusters);
  cfg.blockDim = dim3(p.indices != nullptr ? kThreads : kDenseThreads);
  cfg.dynamicSmemBytes = kSmemAlloc;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (p.indices == nullptr && narrow_decode_shape(p.s_q, p.h_q, p.batch, p.max_pages, num_clusters))
    return launch_decode_narrow(m.kv_lat, p, num_clusters, stream);
  if (p.indices != nullptr)
    return cudaLaunchKernelEx(&cfg, mla_decode_kernel<true>, m.q_rope, m.kv_lat, m.kv_rope, p);
  return cudaLaunchKernelEx(&cfg, mla_decode_kernel<false>, m.q_rope, m.kv_lat, m.kv_rope, p);
}

}  // namespace mla
