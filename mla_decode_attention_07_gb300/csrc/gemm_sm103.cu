// Tensor-core GEMM for sm_103a (GB300), and the two steps that prepare an
// MLA decode call: the new tokens' rows appended to the paged cache, and the
// query absorbed through W_UK (a GEMM batched over heads).
//
// What the GEMM computes: C[m][n] = sum_k A[m][k] * B[k][n], A K-contiguous
// and B N-contiguous, fp16 or bf16 inputs, fp32 accumulation on the tensor
// cores, C stored as fp16, bf16 (round to nearest even) or fp32.  The GEMM
// tutorial summary ("Designing high-performance GPU kernels with TileLang:
// Tensor-Core GEMM", its comparison table) measures exactly this product in
// FP16 at 2048 x 2048 x 2048 against cuBLAS.
//
// GEMM design for GB300:
//  * One CTA per SM, persistent over 128 x 256 output tiles.  Warp 0 issues
//    the TMA loads (one elected lane), warp 1 owns TMEM and issues the MMAs
//    (one elected lane of the converged warp), warps 2-5 drain accumulators
//    (warp w reaches TMEM lanes [32 (w % 4), +32), so the four cover all 128
//    rows).
//  * A four-stage shared-memory ring of 48 KB: A as a 128 x 64 box and B as
//    four 64 x 64 boxes, all with the 128-byte swizzle; A is the K-major
//    operand, B the MN-major one, so neither is transposed in memory.
//  * Each K-stage is four tcgen05.mma M=128 N=256 K=16 into one of two
//    256-column TMEM accumulators: the epilogue of a tile overlaps the
//    loads and MMAs of the next.
//  * Every wait is bounded (2 s on %globaltimer): on expiry the kernel
//    records MLA_ERR_DEVICE_TIMEOUT, lets in-flight copies and MMAs land,
//    frees TMEM and returns.  No trap.
//
// DeepSeek MLA's query absorption, q[r][h][0:512] = q_nope[r][h][:] W_UK[h]
// (d_nope 128 -> d_c 512 per head) with q[r][h][512:576] = q_rope[r][h][:],
// has its own kernel (mla_absorb_kernel, below).  A decode step has few
// query rows per head (16 at batch 16), so the product is taken transposed,
// q_latent^T = W_UK[h]^T q_nope^T: the 512 latent dims are the MMA's M (four
// 128-row blocks) and the query rows its N (a multiple of 16, at most 128 per
// tile), and no MMA row is spent on padding.  One CTA per (head, row tile);
// W_UK[h] (128 KB) lands as eight 64-dim x 128-row boxes (the MN-major A
// operand, 128-byte swizzle, read as stored) behind one barrier per M block,
// so the first block's MMAs run while the rest arrive; the rows' q_nope is
// the K-major B operand.  Its epilogue has one latent dim per thread (the
// TMEM lane): a warp stores 32 consecutive dims (64 bytes) of a row at a
// time, and copies the rows' rotary parts beside them.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "mla.h"
#include "mla_internal.h"
#include "ptx_sm103.cuh"

namespace mla {
namespace {

constexpr int kGemmThreads = 192;
constexpr int kBM = 128, kBN = 256, kBK = 64;
constexpr int kGStages = 4;
constexpr uint32_t kABytes = kBM * kBK * 2;          // 16 KB
constexpr uint32_t kBBoxBytes = kBK * 64 * 2;        // 8 KB: 64 K-rows x 64 N
constexpr uint32_t kGStageBytes = kABytes + 4 * kBBoxBytes;   // 48 KB
constexpr uint32_t kGBar = kGStages * kGStageBytes;
// barriers: FULL[stages], EMPTY[stages], ACC_FULL[2], ACC_EMPTY[2]
constexpr int G_FULL = 0, G_EMPTY = kGStages, G_ACC_FULL = 2 * kGStages,
              G_ACC_EMPTY = 2 * kGStages + 2, G_COUNT = 2 * kGStages + 4;
constexpr uint32_t kGMisc = kGBar + 8 * G_COUNT;     // TMEM address slot, abort flag
constexpr uint32_t kGSmem = kGMisc + 16 + 1024;      // + slack for 1024-byte alignment
constexpr uint32_t kGTmemCols = 512;
constexpr uint64_t kGWaitNs = 2000000000ull;
constexpr uint64_t kGDrainNs = 2000000ull;
static_assert(kGSmem <= 232448, "shared memory");

struct GemmArgs {
  void* c;
  long long ldc, c_batch;   // elements
  int M, N, K, batch, tiles_m, tiles_n;
  int out_type;             // MLA_DTYPE_F16 / BF16 / F32
  int c_v8;                 // C's base and strides allow 32-byte stores
  int* err;
};

struct GCtx {
  uint32_t sbase, abort_addr;
  int* err;
  __device__ __forceinline__ uint32_t bar(int i) const { return sbase + kGBar + 8u * i; }
};

// Bounded wait for the phase with parity `parity`.
__device__ __forceinline__ bool gwait(const GCtx& x, uint32_t bar, uint32_t parity) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = ptx::globaltimer();
  for (uint32_t i = 1;; ++i) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    if ((i & 63u) == 0u) {
      if (ptx::ld_shared_u32_volatile(x.abort_addr) != 0u) return false;
      if (ptx::globaltimer() - t0 > kGWaitNs) {
        atomicCAS(x.err, 0, MLA_ERR_DEVICE_TIMEOUT);
        ptx::st_shared_u32(x.abort_addr, 1u);
        return false;
      }
    }
  }
}
// Decided for the whole warp, so that warp-collective tcgen05 instructions
// after it are reached by all lanes or none.
__device__ __forceinline__ bool gwait_warp(const GCtx& x, uint32_t bar, uint32_t parity) {
  return __all_sync(0xffffffffu, gwait(x, bar, parity));
}

// 32 accumulator columns of one row to C[row][n0 .. n0 + 32), masked at N.
__device__ __forceinline__ void store_row32(const GemmArgs& a, char* crow, int n0,
                                            const uint32_t (&v)[32]) {
  if (a.out_type == MLA_DTYPE_F32) {
    float* dst = reinterpret_cast<float*>(crow) + n0;
    if (n0 + 32 <= a.N && a.c_v8) {
#pragma unroll
      for (int j = 0; j < 4; ++j)
        ptx::st_global_v8(dst + 8 * j, v[8 * j], v[8 * j + 1], v[8 * j + 2], v[8 * j + 3],
                          v[8 * j + 4], v[8 * j + 5], v[8 * j + 6], v[8 * j + 7]);
    } else if (n0 + 32 <= a.N) {
#pragma unroll
      for (int j = 0; j < 8; ++j)
        reinterpret_cast<float4*>(dst)[j] =
            make_float4(__uint_as_float(v[4 * j]), __uint_as_float(v[4 * j + 1]),
                        __uint_as_float(v[4 * j + 2]), __uint_as_float(v[4 * j + 3]));
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (n0 + j < a.N) dst[j] = __uint_as_float(v[j]);
    }
    return;
  }
  uint32_t p[16];
  if (a.out_type == MLA_DTYPE_BF16) {
#pragma unroll
    for (int j = 0; j < 16; ++j)
      p[j] = ptx::pack_bf16x2(__uint_as_float(v[2 * j]), __uint_as_float(v[2 * j + 1]));
  } else {
#pragma unroll
    for (int j = 0; j < 16; ++j)
      p[j] = ptx::pack_f16x2(__uint_as_float(v[2 * j]), __uint_as_float(v[2 * j + 1]));
  }
  uint16_t* dst = reinterpret_cast<uint16_t*>(crow) + n0;
  if (n0 + 32 <= a.N && a.c_v8) {
    // a row's 64 bytes in two 32-byte stores (rows lie ldc apart: whole
    // sectors per store)
    ptx::st_global_v8(dst, p[0], p[1], p[2], p[3], p[4], p[5], p[6], p[7]);
    ptx::st_global_v8(dst + 16, p[8], p[9], p[10], p[11], p[12], p[13], p[14], p[15]);
  } else if (n0 + 32 <= a.N) {
#pragma unroll
    for (int j = 0; j < 4; ++j)
      reinterpret_cast<uint4*>(dst)[j] = make_uint4(p[4 * j], p[4 * j + 1], p[4 * j + 2], p[4 * j + 3]);
  } else {
#pragma unroll
    for (int j = 0; j < 32; ++j)
      if (n0 + j < a.N) dst[j] = (uint16_t)((j & 1) ? (p[j >> 1] >> 16) : (p[j >> 1] & 0xffffu));
  }
}

template <int kInBf16>
__global__ void __launch_bounds__(kGemmThreads, 1)
    mla_gemm_kernel(const __grid_constant__ CUtensorMap tm_a,
                    const __grid_constant__ CUtensorMap tm_b, const GemmArgs args) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  GCtx x;
  x.sbase = (ptx::smem_addr(smem_raw) + 1023u) & ~1023u;
  x.abort_addr = x.sbase + kGMisc + 4;
  x.err = args.err;
  const uint32_t tslot = x.sbase + kGMisc;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kGStages; ++s) {
      ptx::mbar_init(x.bar(G_FULL + s), 1);    // the producer's expect_tx (+ TMA bytes)
      ptx::mbar_init(x.bar(G_EMPTY + s), 1);   // MMA commit
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(x.bar(G_ACC_FULL + a), 1);    // MMA commit
      ptx::mbar_init(x.bar(G_ACC_EMPTY + a), 4);   // the four epilogue warps
    }
    ptx::st_shared_u32(x.abort_addr, 0u);
    ptx::fence_mbarrier_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc(tslot, kGTmemCols);
    ptx::tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    ptx::prefetch_tmap(&tm_a);
    ptx::prefetch_tmap(&tm_b);
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = ptx::ld_shared_u32_volatile(tslot);
  // Launched as a programmatic dependent of the previous kernel on the
  // stream: the set-up above overlaps its tail; its results (A, B) and its
  // use of C are safe once it has completed.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  const int total = args.batch * args.tiles_m * args.tiles_n;
  const int kb_n = (args.K + kBK - 1) / kBK;

  if (warp == 0) {
    // TMA producer
    if (lane == 0) {
      uint32_t it = 0;
      bool ok = true;
      for (int t = blockIdx.x; ok && t < total; t += gridDim.x) {
        const int nt = t % args.tiles_n, rest = t / args.tiles_n;
        const int mt = rest % args.tiles_m, b = rest / args.tiles_m;
        for (int kb = 0; kb < kb_n; ++kb, ++it) {
          const uint32_t s = it % kGStages, ph = (it / kGStages) & 1u;
          if (!gwait(x, x.bar(G_EMPTY + s), ph ^ 1u)) {
            ok = false;
            break;
          }
          ptx::mbar_arrive_expect_tx(x.bar(G_FULL + s), kGStageBytes);
          const uint32_t st = x.sbase + s * kGStageBytes;
          ptx::tma_load_3d(st, &tm_a, kb * kBK, b, mt * kBM, x.bar(G_FULL + s));
#pragma unroll
          for (int j = 0; j < 4; ++j)
            ptx::tma_load_3d(st + kABytes + j * kBBoxBytes, &tm_b, nt * kBN + 64 * j, kb * kBK, b,
                             x.bar(G_FULL + s));
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // MMA issuer: A K-major, B MN-major, both 128-byte swizzled.  A K-step of
    // 16 is 32 bytes into A's rows and 16 rows (2 KB) down B's boxes; B's
    // 64-column boxes are 8 KB apart.
    constexpr uint32_t idesc = ptx::idesc_f32acc(kBM, kBN, 0, 1, kInBf16);
    uint32_t it = 0, lt = 0;
    bool ok = true;
    for (int t = blockIdx.x; ok && t < total; t += gridDim.x, ++lt) {
      const uint32_t acc = lt & 1u;
      if (!gwait_warp(x, x.bar(G_ACC_EMPTY + acc), ((lt >> 1) & 1u) ^ 1u)) {
        ok = false;
        break;
      }
      ptx::tc_fence_after();
      const uint32_t d = tmem + acc * (uint32_t)kBN;
      for (int kb = 0; kb < kb_n; ++kb, ++it) {
        const uint32_t s = it % kGStages, ph = (it / kGStages) & 1u;
        if (!gwait_warp(x, x.bar(G_FULL + s), ph)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t st = x.sbase + s * kGStageBytes;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint64_t ad = ptx::smem_desc(st + k * 32, 16, 1024, ptx::kLayoutSw128);
          const uint64_t bd = ptx::smem_desc(st + kABytes + k * 2048, kBBoxBytes, 1024,
                                             ptx::kLayoutSw128);
          ptx::mma_ss_elect(d, ad, bd, idesc, (kb | k) ? 1u : 0u);
        }
        ptx::mma_commit_elect(x.bar(G_EMPTY + s));
      }
      if (ok) ptx::mma_commit_elect(x.bar(G_ACC_FULL + acc));
    }
    __syncwarp();
  } else {
    // Epilogue: TMEM -> registers -> C, one row per thread.
    const int quad = warp & 3;
    uint32_t lt = 0;
    for (int t = blockIdx.x; t < total; t += gridDim.x, ++lt) {
      const int nt = t % args.tiles_n, rest = t / args.tiles_n;
      const int mt = rest % args.tiles_m, b = rest / args.tiles_m;
      const uint32_t acc = lt & 1u;
      const int row = mt * kBM + quad * 32 + lane;
      if (!gwait_warp(x, x.bar(G_ACC_FULL + acc), (lt >> 1) & 1u)) break;
      ptx::tc_fence_after();
      const int esize = args.out_type == MLA_DTYPE_F32 ? 4 : 2;
      char* crow = static_cast<char*>(args.c) +
                   ((long long)b * args.c_batch + (long long)row * args.ldc) * esize;
#pragma unroll 1
      for (int ch = 0; ch < kBN / 32; ++ch) {
        uint32_t v[32];
        ptx::tmem_ld32_wait(tmem + ((uint32_t)(quad * 32) << 16) + acc * (uint32_t)kBN + ch * 32, v);
        const int n0 = nt * kBN + ch * 32;
        if (row < args.M && n0 < args.N) store_row32(args, crow, n0, v);
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(x.bar(G_ACC_EMPTY + acc));
    }
  }

  // Teardown: after an abort, let in-flight copies and MMAs land before the
  // shared memory and TMEM are released.
  __syncthreads();
  if (ptx::ld_shared_u32_volatile(x.abort_addr) != 0u) {
    const uint64_t t0 = ptx::globaltimer();
    while (ptx::globaltimer() - t0 < kGDrainNs) __nanosleep(1000);
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kGTmemCols);
  }
}

// The new tokens' rows into the paged cache: 16-byte piece c of row (b, i)
// goes to slot t % 64 of page block_table[b][t / 64], t = L_b - s_q + i.
__global__ void mla_cache_append_kernel(const uint4* __restrict__ kv_new, uint4* __restrict__ kv,
                                        int num_pages, const int32_t* __restrict__ block_table,
                                        int max_pages, const int32_t* __restrict__ seqlens,
                                        int s_q, long long pieces, int* err) {
  asm volatile("griddepcontrol.wait;" ::: "memory");   // as in mla_gemm_kernel
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < pieces;
       i += (long long)gridDim.x * blockDim.x) {
    const long long row = i / 72;
    const int c = (int)(i - row * 72);
    const int b = (int)(row / s_q), k = (int)(row - (long long)b * s_q);
    const int t = seqlens[b] - s_q + k;
    if (t < 0 || t / kPageTokens >= max_pages) {
      atomicCAS(err, 0, MLA_ERR_DEVICE_BOUNDS);
      continue;
    }
    const int page = block_table[(long long)b * max_pages + t / kPageTokens];
    if ((unsigned)page >= (unsigned)num_pages) {
      atomicCAS(err, 0, MLA_ERR_DEVICE_BOUNDS);
      continue;
    }
    kv[((long long)page * kPageTokens + t % kPageTokens) * 72 + c] = kv_new[i];
  }
}


// ------------------------------------------------------------ absorption
constexpr int kAbsNope = 128, kAbsC = 512;
constexpr int kAbsMaxN = 128;                          // query rows per tile (TMEM: 4 x N columns)
constexpr uint32_t kAbsWBox = 64 * kAbsNope * 2;      // 16 KB: 64 latent dims x 128 d_nope rows
constexpr uint32_t kAbsQOff = 8 * kAbsWBox;            // 128 KB of W_UK[h], then the q_nope tile
constexpr uint32_t kAbsStage = kAbsQOff + 2 * kAbsMaxN * 128;   // two output staging tiles
constexpr uint32_t kAbsBar = kAbsStage + 2 * (2 * kAbsMaxN * 128);
// barriers: FULL[4] (one per M block; block 0 also counts the q_nope tile),
// SFREE (the MMAs are done with the operands), ACC_FULL[4] (M block m's
// accumulator is complete, so the epilogue drains it while later blocks'
// operands still land), ACC_EMPTY
constexpr int AB_FULL = 0, AB_SFREE = 4, AB_ACC_FULL = 5, AB_ACC_EMPTY = 9, AB_COUNT = 10;
constexpr uint32_t kAbsMisc = kAbsBar + 8 * AB_COUNT;
constexpr uint32_t kAbsSmem = kAbsMisc + 16 + 1024;
static_assert(kAbsSmem <= 232448, "shared memory");

struct AbsorbArgs {
  uint16_t* q;              // bf16 [rows][heads][576]
  const uint4* rope;        // bf16 [rows][heads][64] as 16-byte pieces
  int rows, heads, n_tiles, nt;
  int* err;
};

__global__ void __launch_bounds__(kGemmThreads, 1)
    mla_absorb_kernel(const __grid_constant__ CUtensorMap tm_w,
                      const __grid_constant__ CUtensorMap tm_q,
                      const __grid_constant__ CUtensorMap tm_out, const AbsorbArgs args) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  GCtx x;
  x.sbase = (ptx::smem_addr(smem_raw) + 1023u) & ~1023u;
  x.abort_addr = x.sbase + kAbsMisc + 4;
  x.err = args.err;
  const uint32_t tslot = x.sbase + kAbsMisc;
  auto bar = [&](int i) { return x.sbase + kAbsBar + 8u * i; };
  const int nt = args.nt;
  const uint32_t qbox = (uint32_t)nt * 128u;          // one 64-deep K box of the row tile

  if (threadIdx.x == 0) {
    for (int m = 0; m < 4; ++m) ptx::mbar_init(bar(AB_FULL + m), 1);
    ptx::mbar_init(bar(AB_SFREE), 1);
    for (int m = 0; m < 4; ++m) ptx::mbar_init(bar(AB_ACC_FULL + m), 1);
    ptx::mbar_init(bar(AB_ACC_EMPTY), 4);
    ptx::st_shared_u32(x.abort_addr, 0u);
    ptx::fence_mbarrier_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc(tslot, kGTmemCols);
    ptx::tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    ptx::prefetch_tmap(&tm_w);
    ptx::prefetch_tmap(&tm_q);
    ptx::prefetch_tmap(&tm_out);
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = ptx::ld_shared_u32_volatile(tslot);
  asm volatile("griddepcontrol.wait;" ::: "memory");   // as in mla_gemm_kernel
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int units = args.heads * args.n_tiles;

  if (warp == 0) {
    // TMA producer: a unit's operands, M block by M block
    if (lane == 0) {
      uint32_t lt = 0;
      for (int u = blockIdx.x; u < units; u += gridDim.x, ++lt) {
        const int h = u / args.n_tiles, j = u - h * args.n_tiles;
        if (!gwait(x, bar(AB_SFREE), (lt & 1u) ^ 1u)) break;
        for (int m = 0; m < 4; ++m) {
          const uint32_t fb = bar(AB_FULL + m);
          ptx::mbar_arrive_expect_tx(fb, 2 * kAbsWBox + (m == 0 ? 2 * qbox : 0u));
          if (m == 0) {
            ptx::tma_load_3d(x.sbase + kAbsQOff, &tm_q, 0, h, j * nt, fb);
            ptx::tma_load_3d(x.sbase + kAbsQOff + qbox, &tm_q, 64, h, j * nt, fb);
          }
          ptx::tma_load_3d(x.sbase + (2 * m) * kAbsWBox, &tm_w, 128 * m, 0, h, fb);
          ptx::tma_load_3d(x.sbase + (2 * m + 1) * kAbsWBox, &tm_w, 128 * m + 64, 0, h, fb);
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // MMA issuer: D[m] (128 latent dims x nt rows) = W^T (MN-major: 64-dim
    // atoms 16 KB apart, 8-row groups 1024 B apart; a K step of 16 is 2 KB
    // down the box) times q_nope^T (K-major, 128-byte swizzled rows).
    const uint32_t idesc = ptx::idesc_bf16_f32(128, nt, 1, 0);
    // one accumulator barrier per M block when every CTA has one unit (the
    // epilogue drains the blocks as they finish), else one for the whole
    // accumulator (extra commits between the blocks cost more than they give
    // when the next unit's MMAs follow)
    const bool per_block = units <= (int)gridDim.x;
    uint32_t lt = 0;
    bool ok = true;
    for (int u = blockIdx.x; ok && u < units; u += gridDim.x, ++lt) {
      if (!gwait_warp(x, bar(AB_ACC_EMPTY), (lt & 1u) ^ 1u)) break;
      ptx::tc_fence_after();
      for (int m = 0; m < 4; ++m) {
        if (!gwait_warp(x, bar(AB_FULL + m), lt & 1u)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
#pragma unroll
        for (int k = 0; k < kAbsNope / 16; ++k) {
          const uint64_t ad = ptx::smem_desc(x.sbase + (2 * m) * kAbsWBox + k * 2048, kAbsWBox,
                                             1024, ptx::kLayoutSw128);
          const uint64_t bd = ptx::smem_desc(x.sbase + kAbsQOff + (k >> 2) * qbox + (k & 3) * 32,
                                             16, 1024, ptx::kLayoutSw128);
          ptx::mma_ss_elect(tmem + (uint32_t)(m * nt), ad, bd, idesc, k > 0 ? 1u : 0u);
        }
        if (per_block) ptx::mma_commit_elect(bar(AB_ACC_FULL + m));
      }
      if (!ok) break;
      // the operands first: the next unit's loads start as early as possible
      ptx::mma_commit_elect(bar(AB_SFREE));
      if (!per_block) ptx::mma_commit_elect(bar(AB_ACC_FULL + 3));
    }
    __syncwarp();
  } else {
    // Epilogue: thread = latent dim 32 * quad + lane of each M block.  A
    // block goes through a shared-memory tile (two 64-dim halves of nt rows
    // x 128 bytes, double-buffered) and out by two TMA tensor stores, which
    // skip the rows past the end; the rows' rotary parts are plain copies.
    const int quad = warp & 3, et = threadIdx.x - 64;
    const long long rstride = (long long)args.heads * kDqk;
    const uint32_t my_col = (uint32_t)(quad >> 1) * qbox + (uint32_t)((quad & 1) * 32 + lane) * 2u;
    // the same choice as the MMA issuer's: per block, or the whole accumulator
    const bool per_block = units <= (int)gridDim.x;
    uint32_t lt = 0, blk = 0;
    for (int u = blockIdx.x; u < units; u += gridDim.x, ++lt) {
      const int h = u / args.n_tiles, j = u - h * args.n_tiles;
      const int row0 = j * nt;
      // the rows' rotary parts (8 pieces a row), loaded before the
      // accumulator wait so that their latency overlaps the MMAs
      uint4 rp[kAbsMaxN / 16];
#pragma unroll
      for (int i = 0; i < kAbsMaxN / 16; ++i) {
        const int pc = et + 128 * i, r = row0 + (pc >> 3);
        if (i < nt / 16 && r < args.rows) rp[i] = args.rope[((long long)r * args.heads + h) * 8 + (pc & 7)];
      }
      // Every epilogue warp comes to the named barrier after an accumulator
      // wait, whether the wait succeeded or not, so the abort decision after
      // it is the same for all four.
      bool aborted = false;
      if (!per_block) {
        gwait_warp(x, bar(AB_ACC_FULL + 3), lt & 1u);
        ptx::named_sync(1, 128);
        aborted = ptx::ld_shared_u32_volatile(x.abort_addr) != 0u;
        ptx::tc_fence_after();
      }
      for (int m = 0; !aborted && m < 4; ++m, ++blk) {
        if (per_block) {
          gwait_warp(x, bar(AB_ACC_FULL + m), lt & 1u);
          ptx::named_sync(1, 128);
          if (ptx::ld_shared_u32_volatile(x.abort_addr) != 0u) {
            aborted = true;
            break;
          }
          ptx::tc_fence_after();
        }
        const uint32_t stg = x.sbase + kAbsStage + (blk & 1u) * 2u * qbox;
        if (et == 0) ptx::bulk_wait_read<1>();   // the store that last read this buffer is done
        ptx::named_sync(1, 128);
        for (int c0 = 0; c0 < nt; c0 += 16) {
          uint32_t v[16];
          ptx::tmem_ld32x16_wait(tmem + ((uint32_t)(quad * 32) << 16) + (uint32_t)(m * nt + c0), v);
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const uint16_t b16 = (uint16_t)(ptx::pack_bf16x2(__uint_as_float(v[i]), 0.f) & 0xffffu);
            asm volatile("st.shared.u16 [%0], %1;" ::"r"(stg + my_col + (uint32_t)(c0 + i) * 128u),
                         "h"(b16)
                         : "memory");
          }
        }
        ptx::fence_proxy_async_smem();
        ptx::named_sync(1, 128);
        if (et == 0) {
          ptx::tma_store_3d(&tm_out, 128 * m, h, row0, stg);
          ptx::tma_store_3d(&tm_out, 128 * m + 64, h, row0, stg + qbox);
          ptx::bulk_commit();
        }
      }
      if (aborted) break;
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(bar(AB_ACC_EMPTY));
#pragma unroll
      for (int i = 0; i < kAbsMaxN / 16; ++i) {
        const int pc = et + 128 * i, r = row0 + (pc >> 3);
        if (i < nt / 16 && r < args.rows)
          reinterpret_cast<uint4*>(args.q + (long long)r * rstride + (long long)h * kDqk + kAbsC)[pc & 7] =
              rp[i];
      }
    }
    if (et == 0) ptx::bulk_wait_all();
  }

  __syncthreads();
  if (ptx::ld_shared_u32_volatile(x.abort_addr) != 0u) {
    const uint64_t t0 = ptx::globaltimer();
    while (ptx::globaltimer() - t0 < kGDrainNs) __nanosleep(1000);
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kGTmemCols);
  }
}

std::once_flag g_gemm_attr_once[64];
cudaError_t g_gemm_attr_status[64];

cudaError_t gemm_setup(int device) {
  if (device < 0 || device >= 64) return cudaErrorInvalidDevice;
  std::call_once(g_gemm_attr_once[device], [&]() {
    cudaError_t e = cudaFuncSetAttribute(mla_gemm_kernel<0>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kGSmem);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(mla_gemm_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)kGSmem);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(mla_absorb_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)kAbsSmem);
    g_gemm_attr_status[device] = e;
  });
  return g_gemm_attr_status[device];
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Launch configuration with programmatic stream serialization: the kernel may
// start while the previous one on the stream finishes, and waits for it
// (griddepcontrol.wait) before touching global memory.
struct PdlLaunch {
  cudaLaunchConfig_t cfg;
  cudaLaunchAttribute attr[1];
  PdlLaunch(int grid, int threads, size_t smem, cudaStream_t stream) {
    cfg = cudaLaunchConfig_t{};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
};

// One batched GEMM launch.  A map: dims {K, batch, M}; B map: {N, K, batch}.
int launch_gemm(int in_dtype, const CUtensorMap& ma, const CUtensorMap& mb, GemmArgs a,
                cudaStream_t stream) {
  int device = 0, sms = 0;
  int* err = nullptr;
  const int st = device_current(&device, &sms, &err);
  if (st != MLA_OK) return st;
  if (gemm_setup(device) != cudaSuccess) return MLA_ERR_CUDA;
  a.err = err;
  a.tiles_m = (a.M + kBM - 1) / kBM;
  a.tiles_n = (a.N + kBN - 1) / kBN;
  const long long total = (long long)a.batch * a.tiles_m * a.tiles_n;
  if (total >= (1ll << 31)) return MLA_ERR_INVALID_ARG;
  const int grid = (int)(total < sms ? total : sms);
  PdlLaunch l(grid, kGemmThreads, kGSmem, stream);
  const cudaError_t e = in_dtype == MLA_DTYPE_BF16
                            ? cudaLaunchKernelEx(&l.cfg, mla_gemm_kernel<1>, ma, mb, a)
                            : cudaLaunchKernelEx(&l.cfg, mla_gemm_kernel<0>, ma, mb, a);
  return e == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

}  // namespace
}  // namespace mla

using namespace mla;

extern "C" {

int mla_gemm(const void* A, const void* B, void* C, int M, int N, int K, int in_dtype,
             int out_dtype, void* stream) {
  if (!A || !B || !C || M < 1 || N < 1 || K < 1 || (N % 8) != 0 || (K % 8) != 0 ||
      (in_dtype != MLA_DTYPE_F16 && in_dtype != MLA_DTYPE_BF16) ||
      (out_dtype != MLA_DTYPE_F16 && out_dtype != MLA_DTYPE_BF16 && out_dtype != MLA_DTYPE_F32) ||
      !aligned16(A) || !aligned16(B) || !aligned16(C))
    return MLA_ERR_INVALID_ARG;
  const CUtensorMapDataType dt =
      in_dtype == MLA_DTYPE_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  CUtensorMap ma, mb;
  const uint64_t da[3] = {(uint64_t)K, 1, (uint64_t)M};
  const uint64_t sa[2] = {(uint64_t)K * 2, (uint64_t)K * 2};
  const uint32_t ba[3] = {kBK, 1, kBM};
  const uint64_t db[3] = {(uint64_t)N, (uint64_t)K, 1};
  const uint64_t sb[2] = {(uint64_t)N * 2, (uint64_t)N * K * 2};
  const uint32_t bb[3] = {64, kBK, 1};
  if (!encode_tiled_map(&ma, dt, 3, A, da, sa, ba, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_tiled_map(&mb, dt, 3, B, db, sb, bb, CU_TENSOR_MAP_SWIZZLE_128B))
    return MLA_ERR_CUDA;
  GemmArgs a = {};
  a.c = C;
  a.ldc = N;
  a.c_batch = (long long)M * N;
  a.M = M;
  a.N = N;
  a.K = K;
  a.batch = 1;
  a.out_type = out_dtype;
  {
    const size_t es = out_dtype == MLA_DTYPE_F32 ? 4 : 2;
    a.c_v8 = (reinterpret_cast<uintptr_t>(C) & 31u) == 0 && ((size_t)N * es) % 32 == 0;
  }
  return launch_gemm(in_dtype, ma, mb, a, static_cast<cudaStream_t>(stream));
}

int mla_q_absorb(const void* q_nope, const void* q_rope, const void* w_uk, void* q, int batch,
                 int s_q, int h_q, void* stream) {
  if (!q_nope || !q_rope || !w_uk || !q || batch < 1 || s_q < 1 || h_q < 1 ||
      (long long)batch * s_q * h_q >= (1ll << 31) || !aligned16(q_nope) || !aligned16(q_rope) ||
      !aligned16(w_uk) || !aligned16(q))
    return MLA_ERR_INVALID_ARG;
  const int rows = batch * s_q;
  // row tiles of equal size, a multiple of 16 and at most 128
  const int n_tiles = (rows + kAbsMaxN - 1) / kAbsMaxN;
  const int nt = ((rows + n_tiles - 1) / n_tiles + 15) / 16 * 16;
  CUtensorMap mw, mq, mo;
  // W_UK [h_q][128][512]: latent dims innermost, d_nope next, heads outermost
  const uint64_t dw[3] = {kAbsC, kAbsNope, (uint64_t)h_q};
  const uint64_t sw[2] = {kAbsC * 2, (uint64_t)kAbsNope * kAbsC * 2};
  const uint32_t bw[3] = {64, kAbsNope, 1};
  // q_nope [rows][h_q][128]: d_nope innermost, heads next, rows outermost
  const uint64_t dq[3] = {kAbsNope, (uint64_t)h_q, (uint64_t)rows};
  const uint64_t sq[2] = {kAbsNope * 2, (uint64_t)h_q * kAbsNope * 2};
  const uint32_t bq[3] = {64, 1, (uint32_t)nt};
  // q [rows][h_q][576] (stored into): dims innermost, heads next, rows outermost
  const uint64_t dout[3] = {kDqk, (uint64_t)h_q, (uint64_t)rows};
  const uint64_t sout[2] = {kDqk * 2, (uint64_t)h_q * kDqk * 2};
  const uint32_t bout[3] = {64, 1, (uint32_t)nt};
  if (!encode_tiled_map(&mw, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, w_uk, dw, sw, bw,
                        CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_tiled_map(&mq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, q_nope, dq, sq, bq,
                        CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_tiled_map(&mo, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, q, dout, sout, bout,
                        CU_TENSOR_MAP_SWIZZLE_NONE))
    return MLA_ERR_CUDA;
  int device = 0, sms = 0;
  int* err = nullptr;
  const int st = device_current(&device, &sms, &err);
  if (st != MLA_OK) return st;
  if (gemm_setup(device) != cudaSuccess) return MLA_ERR_CUDA;
  AbsorbArgs a;
  a.q = static_cast<uint16_t*>(q);
  a.rope = static_cast<const uint4*>(q_rope);
  a.rows = rows;
  a.heads = h_q;
  a.n_tiles = n_tiles;
  a.nt = nt;
  a.err = err;
  const long long units = (long long)h_q * n_tiles;
  if (units >= (1ll << 31)) return MLA_ERR_INVALID_ARG;
  const int grid = (int)(units < sms ? units : sms);
  PdlLaunch l(grid, kGemmThreads, kAbsSmem, static_cast<cudaStream_t>(stream));
  return cudaLaunchKernelEx(&l.cfg, mla_absorb_kernel, mw, mq, mo, a) == cudaSuccess ? MLA_OK
                                                                                      : MLA_ERR_CUDA;
}

int mla_cache_append(const void* kv_new, void* kv_cache, int num_pages, const int32_t* block_table,
                     int max_pages, const int32_t* cache_seqlens, int batch, int s_q,
                     void* stream) {
  if (!kv_new || !kv_cache || !block_table || !cache_seqlens || batch < 1 || s_q < 1 ||
      num_pages < 1 || max_pages < 1 || (long long)num_pages * kPageTokens >= (1ll << 31) ||
      !aligned16(kv_new) || !aligned16(kv_cache) ||
      (reinterpret_cast<uintptr_t>(block_table) & 3u) || (reinterpret_cast<uintptr_t>(cache_seqlens) & 3u))
    return MLA_ERR_INVALID_ARG;
  int device = 0, sms = 0;
  int* err = nullptr;
  const int st = device_current(&device, &sms, &err);
  if (st != MLA_OK) return st;
  const long long pieces = (long long)batch * s_q * 72;
  const int grid = (int)((pieces + 255) / 256 < 2 * sms ? (pieces + 255) / 256 : 2 * sms);
  PdlLaunch l(grid, 256, 0, static_cast<cudaStream_t>(stream));
  return cudaLaunchKernelEx(&l.cfg, mla_cache_append_kernel, static_cast<const uint4*>(kv_new),
                            static_cast<uint4*>(kv_cache), num_pages, block_table, max_pages,
                            cache_seqlens, s_q, pieces, err) == cudaSuccess
             ? MLA_OK
             : MLA_ERR_CUDA;
}

}  // extern "C"
