// libmla C ABI: argument checks, tensor maps, the split-KV planner kernel,
// the LSE-combine kernel, and the device error word.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

#include <mutex>

#include "mla.h"
#include "mla_internal.h"
#include "ptx_sm103.cuh"

namespace mla {
namespace {

__device__ int g_device_error;   // first device-side error of any launch, 0 if none

constexpr int kMaxDevices = 64;
constexpr int kPlanThreads = 256;
constexpr int kCombineWarps = 8;

// ------------------------------------------------------------------ planner
// Exclusive prefix sum over the CTA; `total` receives the CTA-wide sum.
__device__ long long block_exclusive_scan(long long v, long long* warp_sums, long long& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  long long x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const long long y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_sums[warp] = x;
  __syncthreads();
  if (warp == 0) {
    long long s = lane < nwarps ? warp_sums[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const long long y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    if (lane < nwarps) warp_sums[lane] = s;
  }
  __syncthreads();
  const long long before = warp == 0 ? 0 : warp_sums[warp - 1];
  total = warp_sums[nwarps - 1];
  __syncthreads();
  return before + x - v;
}

// The unit prefix sums are searched many times (two binary searches per
// cluster, two lookups per batch entry); they and the page counts live in
// shared memory when they fit (kPlanSmemBatch entries), in the plan buffer
// otherwise.
constexpr int kPlanSmemBatch = 4000;

__global__ void __launch_bounds__(kPlanThreads) mla_plan_kernel(const int32_t* seqlens, int batch,
                                                                int s_q, int h_q, int num_clusters,
                                                                int32_t* plan, int* err) {
  __shared__ long long warp_sums[32];
  extern __shared__ int64_t starts_smem[];
  // The decode kernel may launch now: it reads the plan only after waiting
  // for this grid to complete.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // This grid is itself launched as a programmatic dependent of whatever
  // precedes it on the stream (typically the previous step's combine, which
  // still reads the plan buffer): wait for it to complete before reading the
  // lengths or writing the plan.  Being launched early hides the launch.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int tiles = plan_tiles(s_q, h_q);
  const int gt = plan_group_clusters(num_clusters, tiles);
  int64_t* starts_g = reinterpret_cast<int64_t*>(reinterpret_cast<char*>(plan) +
                                                 plan_off_starts(batch, gt));
  const bool in_smem = batch <= kPlanSmemBatch;
  int64_t* starts = in_smem ? starts_smem : starts_g;
  int32_t* items = plan + plan_off_items(gt) / 4;
  int32_t* pages = in_smem ? reinterpret_cast<int32_t*>(starts_smem + batch + 1) : items;
  const int pstride = in_smem ? 1 : kItemWords;
  int32_t* clus = plan + H_WORDS;

  // 1. unit intervals of the batch entries
  long long run = 0;
  for (int base = 0; base < batch; base += blockDim.x) {
    const int b = base + threadIdx.x;
    int L = b < batch ? seqlens[b] : 0;
    if (L < 0) {
      atomicCAS(err, 0, MLA_ERR_DEVICE_BOUNDS);
      L = 0;
    }
    const int P = pages_of(L);
    long long tot;
    const long long ex = block_exclusive_scan(units_of(P), warp_sums, tot);
    if (b < batch) {
      starts[b] = run + ex;
      starts_g[b] = run + ex;
      items[b * kItemWords + 0] = P;
      pages[b * pstride] = P;
    }
    run += tot;
  }
  if (threadIdx.x == 0) {
    starts[batch] = run;
    starts_g[batch] = run;
  }
  __syncthreads();
  const long long V = run;
  const int g = plan_used_clusters(V, gt);

  // 2. cluster ranges
  for (int c = threadIdx.x; c < gt; c += blockDim.x) {
    int b0 = batch, p0 = 0, b1 = batch, p1 = 0, s0 = 0;
    if (c < g) {
      cursor_of(starts, batch, cluster_begin(c, V, g), &b0, &p0);
      cursor_of(starts, batch, cluster_begin(c + 1, V, g), &b1, &p1);
      if (b0 < batch) s0 = c - cluster_of(starts[b0] + kSplitOverhead, V, g);
    }
    int32_t* e = clus + c * kClusterWords;
    e[0] = b0;
    e[1] = p0;
    e[2] = b1;
    e[3] = p1;
    e[4] = s0;
    e[5] = 0;
    e[6] = 0;
    e[7] = 0;
  }

  // 3. splits per batch entry and where their partials go
  run = 0;
  for (int base = 0; base < batch; base += blockDim.x) {
    const int b = base + threadIdx.x;
    int ns = 0, cf = -1;
    if (b < batch) {
      const int P = pages[b * pstride];
      if (P > 0) {
        cf = cluster_of(starts[b] + kSplitOverhead, V, g);
        const int cl = cluster_of(starts[b] + kSplitOverhead + P - 1, V, g);
        ns = cl - cf + 1;
      }
    }
    long long tot;
    const long long ex = block_exclusive_scan(ns >= 2 ? ns : 0, warp_sums, tot);
    if (b < batch) {
      items[b * kItemWords + 1] = ns;
      items[b * kItemWords + 2] = (int)(run + ex);
      items[b * kItemWords + 3] = cf;
    }
    run += tot;
  }
  if (threadIdx.x == 0) {
    plan[H_MAGIC] = kPlanMagic;
    plan[H_BATCH] = batch;
    plan[H_SQ] = s_q;
    plan[H_HQ] = h_q;
    plan[H_TILES] = tiles;
    plan[H_GT] = gt;
    plan[H_GUSED] = g;
    plan[H_STOTAL] = (int)run;
    plan[H_OVH] = kSplitOverhead;
    plan[H_NCLUSTERS] = num_clusters;
    for (int k = H_NCLUSTERS + 1; k < H_WORDS; ++k) plan[k] = 0;
  }
}

// Host mirror of mla_plan_kernel: the same integer formulas, in order.
void plan_host(const int32_t* seqlens, int batch, int s_q, int h_q, int num_clusters,
               int32_t* plan) {
  const int tiles = plan_tiles(s_q, h_q);
  const int gt = plan_group_clusters(num_clusters, tiles);
  int64_t* starts = reinterpret_cast<int64_t*>(reinterpret_cast<char*>(plan) +
                                               plan_off_starts(batch, gt));
  int32_t* items = plan + plan_off_items(gt) / 4;
  int32_t* clus = plan + H_WORDS;
  int64_t run = 0;
  for (int b = 0; b < batch; ++b) {
    const int L = seqlens[b] < 0 ? 0 : seqlens[b];
    const int P = pages_of(L);
    starts[b] = run;
    items[b * kItemWords + 0] = P;
    run += units_of(P);
  }
  starts[batch] = run;
  const int64_t V = run;
  const int g = plan_used_clusters(V, gt);
  for (int c = 0; c < gt; ++c) {
    int b0 = batch, p0 = 0, b1 = batch, p1 = 0, s0 = 0;
    if (c < g) {
      cursor_of(starts, batch, cluster_begin(c, V, g), &b0, &p0);
      cursor_of(starts, batch, cluster_begin(c + 1, V, g), &b1, &p1);
      if (b0 < batch) s0 = c - cluster_of(starts[b0] + kSplitOverhead, V, g);
    }
    int32_t* e = clus + c * kClusterWords;
    e[0] = b0;
    e[1] = p0;
    e[2] = b1;
    e[3] = p1;
    e[4] = s0;
    e[5] = e[6] = e[7] = 0;
  }
  int64_t sb = 0;
  for (int b = 0; b < batch; ++b) {
    int ns = 0, cf = -1;
    const int P = items[b * kItemWords + 0];
    if (P > 0) {
      cf = cluster_of(starts[b] + kSplitOverhead, V, g);
      const int cl = cluster_of(starts[b] + kSplitOverhead + P - 1, V, g);
      ns = cl - cf + 1;
    }
    items[b * kItemWords + 1] = ns;
    items[b * kItemWords + 2] = (int)sb;
    items[b * kItemWords + 3] = cf;
    sb += ns >= 2 ? ns : 0;
  }
  plan[H_MAGIC] = kPlanMagic;
  plan[H_BATCH] = batch;
  plan[H_SQ] = s_q;
  plan[H_HQ] = h_q;
  plan[H_TILES] = tiles;
  plan[H_GT] = gt;
  plan[H_GUSED] = g;
  plan[H_STOTAL] = (int)sb;
  plan[H_OVH] = kSplitOverhead;
  plan[H_NCLUSTERS] = num_clusters;
  for (int k = H_NCLUSTERS + 1; k < H_WORDS; ++k) plan[k] = 0;
}

// ------------------------------------------------------------------ combine
// Merges the split partials of every (batch entry, tile) that has two or
// more splits:  lse = m + ln(sum_j exp(lse_j - m)),  out = sum_j
// exp(lse_j - lse) * o_j.  Entries without pages get out = 0, lse = -inf.
// The decode kernel stores partials as [slot][dim/4][row][4] fp32, so one
// job (a batch entry's tile and 16 of its dims) reads, per split, 128 rows x
// 2 x 16 bytes per half of its threads, every warp access 512 contiguous
// bytes.  All of a job's loads (the split lse values and partial outputs, up
// to kCombineBatch splits at a time) are issued before the first use: the
// job costs about one memory latency after its plan entry is read.
constexpr int kCombineQuads = 4;    // dim groups (of 4) per job

// BATCH splits loaded together; MINB CTAs per SM (the register budget that
// allows).  Six splits at three CTAs per SM, or four at four: the launch picks
// the form that runs its jobs in fewer waves.
template <int BATCH, int MINB>
__global__ void __launch_bounds__(kCombineWarps * 32, MINB) mla_combine_kernel(const DecodeParams p) {
  constexpr int kCombineBatch = BATCH;
  // Launched as a programmatic dependent of the decode kernel, whose blocks
  // let this grid launch only after their own wait on the planner had
  // returned: the plan is complete and visible here, so it is read (past L1)
  // before the wait.  The partials are not, and no output is written before
  // the wait; every block waits once, so that this grid completes only after
  // the decode kernel has.  One thread per block reads the plan words into
  // shared memory: every block reads the same few words, and one L2 request
  // per block instead of one per warp keeps that line from becoming a hot
  // spot.
  // The next kernel on the stream (the next call's main kernel) may launch
  // now: it waits for this grid to complete before it reads anything, and
  // meanwhile its set-up (barriers, TMEM, cluster sync) overlaps this grid.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int32_t* plan = p.plan;
  __shared__ int s_hdr[4];
  __shared__ int s_item[2];
  if (threadIdx.x == 0) {
    s_hdr[0] = __ldcg(plan + H_TILES);
    s_hdr[1] = __ldcg(plan + H_GT);
    s_hdr[2] = __ldcg(plan + H_STOTAL);
    s_hdr[3] = __ldcg(plan + H_NCLUSTERS);
  }
  __syncthreads();
  const int tiles = s_hdr[0], gt = s_hdr[1], stotal = s_hdr[2];
  const int32_t* items = plan + plan_off_items(gt) / 4;
  const int64_t max_slots = workspace_slots(s_hdr[3]);
  bool waited = false;
  const int rows = p.s_q * p.h_q;
  constexpr int kQuadBlocks = (kDv / 4) / kCombineQuads;   // 32
  const int r = threadIdx.x & (kTileRows - 1);             // tile row of this thread
  const int qpair = threadIdx.x >> 7;                      // dim groups 2 qpair, 2 qpair + 1
  const int64_t total = (int64_t)p.batch * tiles * kQuadBlocks;
  for (int64_t job = blockIdx.x; job < total; job += gridDim.x) {
    const int qb = (int)(job % kQuadBlocks);
    const int64_t item = job / kQuadBlocks;
    const int b = (int)(item % p.batch), t = (int)(item / p.batch);
    __syncthreads();                                         // the last job's s_item is read
    if (threadIdx.x == 0) {
      s_item[0] = __ldcg(items + b * kItemWords + 1);
      s_item[1] = __ldcg(items + b * kItemWords + 2);
    }
    __syncthreads();
    const int ns = s_item[0];
    if (ns == 1) continue;                                   // written by the main kernel
    if (t * kTileRows >= rows) continue;                      // padding tile
    const int64_t slot0 = (int64_t)t * stotal + s_item[1];
    if (ns > 1 && (slot0 < 0 || slot0 + ns > max_slots)) {
      if (threadIdx.x == 0) atomicCAS(p.err, 0, MLA_ERR_PLAN);
      continue;
    }
    if (!waited) {
      asm volatile("griddepcontrol.wait;" ::: "memory");
      waited = true;
    }
    const int qr = t * kTileRows + r;
    const float* lse_col = p.ws_lse + slot0 * kTileRows + r;
    const float4* o_col = reinterpret_cast<const float4*>(p.ws_o) + slot0 * (kSlotFloats / 4) +
                          (int64_t)(qb * kCombineQuads + 2 * qpair) * kTileRows + r;
    // running merge over batches of splits (one batch in practice)
    float m = -INFINITY, se = 0.f;
    float4 acc0 = make_float4(0.f, 0.f, 0.f, 0.f), acc1 = acc0;
    for (int c0 = 0; c0 < ns; c0 += kCombineBatch) {
      const int nc = ns - c0 < kCombineBatch ? ns - c0 : kCombineBatch;
      float lj[kCombineBatch];
      float4 v0[kCombineBatch], v1[kCombineBatch];
#pragma unroll
      for (int j = 0; j < kCombineBatch; ++j) {
        if (j < nc) {
          const int64_t s = c0 + j;
          lj[j] = __ldcs(lse_col + s * kTileRows);
          v0[j] = __ldcs(o_col + s * (kSlotFloats / 4));
          v1[j] = __ldcs(o_col + s * (kSlotFloats / 4) + kTileRows);
        } else {
          lj[j] = -INFINITY;
          v0[j] = v1[j] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
      float mb = m;
#pragma unroll
      for (int j = 0; j < kCombineBatch; ++j) mb = fmaxf(mb, lj[j]);
      if (mb == -INFINITY) continue;                          // nothing visible yet
      // rescale what was merged so far to the new max
      const float sc = (m == -INFINITY) ? 0.f : expf(m - mb);
      se *= sc;
      acc0.x *= sc; acc0.y *= sc; acc0.z *= sc; acc0.w *= sc;
      acc1.x *= sc; acc1.y *= sc; acc1.z *= sc; acc1.w *= sc;
      m = mb;
#pragma unroll
      for (int j = 0; j < kCombineBatch; ++j) {
        const float wj = (j < nc) ? expf(lj[j] - m) : 0.f;
        se += wj;
        acc0.x += wj * v0[j].x;
        acc0.y += wj * v0[j].y;
        acc0.z += wj * v0[j].z;
        acc0.w += wj * v0[j].w;
        acc1.x += wj * v1[j].x;
        acc1.y += wj * v1[j].y;
        acc1.z += wj * v1[j].z;
        acc1.w += wj * v1[j].w;
      }
    }
    if (qr >= rows) continue;
    float lse = -INFINITY;
    if (m != -INFINITY) {
      const float inv = 1.0f / se;
      acc0.x *= inv; acc0.y *= inv; acc0.z *= inv; acc0.w *= inv;
      acc1.x *= inv; acc1.y *= inv; acc1.z *= inv; acc1.w *= inv;
      lse = m + logf(se);
    }
    const int i = qr / p.h_q, h = qr - i * p.h_q;
    const int64_t oidx = (((int64_t)b * p.s_q + i) * p.h_q + h) * kDv +
                         (qb * kCombineQuads + 2 * qpair) * 4;
    if (qb == 0 && qpair == 0) p.lse[((int64_t)b * p.h_q + h) * p.s_q + i] = lse;
    if (p.out_f32) {
      float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.out) + oidx);
      dst[0] = acc0;
      dst[1] = acc1;
      continue;
    }
    uint4 u;
    const __nv_bfloat162 a0 = __floats2bfloat162_rn(acc0.x, acc0.y);
    const __nv_bfloat162 a1 = __floats2bfloat162_rn(acc0.z, acc0.w);
    const __nv_bfloat162 a2 = __floats2bfloat162_rn(acc1.x, acc1.y);
    const __nv_bfloat162 a3 = __floats2bfloat162_rn(acc1.z, acc1.w);
    memcpy(&u.x, &a0, 4);
    memcpy(&u.y, &a1, 4);
    memcpy(&u.z, &a2, 4);
    memcpy(&u.w, &a3, 4);
    *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.out) + oidx) = u;
  }
  if (!waited) asm volatile("griddepcontrol.wait;" ::: "memory");
}

// ------------------------------------------------------------------ device state
struct DeviceState {
  std::once_flag once;
  int status = MLA_ERR_CUDA;  // MLA_OK once set up
  int num_sms = 0;
  int num_clusters = 0;
  int* err = nullptr;         // address of g_device_error on this device
};
DeviceState g_dev[kMaxDevices];

int setup_device(int device) {
  if (device < 0 || device >= kMaxDevices) return MLA_ERR_INVALID_ARG;
  DeviceState& d = g_dev[device];
  std::call_once(d.once, [&]() {
    int prev = 0;
    if (cudaGetDevice(&prev) != cudaSuccess) return;
    if (prev != device && cudaSetDevice(device) != cudaSuccess) return;
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, device) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, device) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess) {
      d.status = MLA_ERR_CUDA;
    } else if (major != 10 || minor != 3) {
      d.status = MLA_ERR_UNSUPPORTED_DEVICE;
    } else {
      void* addr = nullptr;
      const int maxc = decode_max_clusters(device);
      if (maxc <= 0 || cudaGetSymbolAddress(&addr, g_device_error) != cudaSuccess) {
        d.status = MLA_ERR_CUDA;
      } else {
        d.num_sms = sms;
        d.num_clusters = maxc < sms / 2 ? maxc : sms / 2;
        d.err = static_cast<int*>(addr);
        d.status = MLA_OK;
      }
    }
    if (prev != device) cudaSetDevice(prev);
  });
  return d.status;
}

bool shape_ok(int batch, int s_q, int h_q) {
  return batch >= 1 && s_q >= 1 && s_q <= 8 && h_q >= 1 && h_q <= 128;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, []() {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

// 2-D bf16 map over [rows, 576] with a (box_cols x box_rows) box.
bool make_map(CUtensorMap* m, const void* base, uint64_t rows, uint32_t box_cols,
              uint32_t box_rows, CUtensorMapSwizzle swz) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)kDqk, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)kDqk * 2};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int64_t workspace_bytes_for(int num_clusters) {
  const int64_t slots = workspace_slots(num_clusters);
  return slots * kSlotFloats * 4 + slots * kTileRows * 4;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

}  // namespace

int device_current(int* device, int* num_sms, int** err) {
  if (cudaGetDevice(device) != cudaSuccess) return MLA_ERR_CUDA;
  const int st = setup_device(*device);
  if (st != MLA_OK) return st;
  *num_sms = g_dev[*device].num_sms;
  *err = g_dev[*device].err;
  return MLA_OK;
}

bool encode_tiled_map(CUtensorMap* m, CUtensorMapDataType dtype, int rank, const void* base,
                      const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box,
                      CUtensorMapSwizzle swz) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
  if (!enc || rank < 1 || rank > 5) return false;
  cuuint64_t d[5], st[4];
  cuuint32_t bx[5], es[5];
  for (int i = 0; i < rank; ++i) {
    d[i] = dims[i];
    bx[i] = box[i];
    es[i] = 1;
    if (i + 1 < rank) st[i] = strides_bytes[i];
  }
  return enc(m, dtype, (cuuint32_t)rank, const_cast<void*>(base), d, st, bx, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace mla

using namespace mla;

extern "C" {

int mla_num_clusters(int device) {
  const int st = setup_device(device);
  return st == MLA_OK ? g_dev[device].num_clusters : st;
}

int mla_decode_kernel_kind(int batch, int s_q, int h_q, int max_pages, int device) {
  if (!shape_ok(batch, s_q, h_q) || max_pages < 1) return MLA_ERR_INVALID_ARG;
  const int st = setup_device(device);
  if (st != MLA_OK) return st;
  return narrow_decode_shape(s_q, h_q, batch, max_pages, g_dev[device].num_clusters) ? 1 : 0;
}

size_t mla_plan_size_for_clusters(int batch, int s_q, int h_q, int num_clusters) {
  if (!shape_ok(batch, s_q, h_q) || num_clusters < 1) return 0;
  const int gt = plan_group_clusters(num_clusters, plan_tiles(s_q, h_q));
  if (gt < 1) return 0;
  return (size_t)plan_bytes(batch, gt);
}

size_t mla_plan_size(int batch, int s_q, int h_q, int device) {
  const int nc = mla_num_clusters(device);
  return nc > 0 ? mla_plan_size_for_clusters(batch, s_q, h_q, nc) : 0;
}

size_t mla_workspace_size(int batch, int s_q, int h_q, int device) {
  if (!shape_ok(batch, s_q, h_q)) return 0;
  const int nc = mla_num_clusters(device);
  return nc > 0 ? (size_t)workspace_bytes_for(nc) : 0;
}

int mla_decode_plan_host(const int32_t* cache_seqlens_host, int batch, int s_q, int h_q,
                         int num_clusters, void* tile_meta_host, size_t tile_meta_bytes) {
  if (!cache_seqlens_host || !tile_meta_host || !shape_ok(batch, s_q, h_q) || num_clusters < 1 ||
      !aligned(tile_meta_host, 8))
    return MLA_ERR_INVALID_ARG;
  const size_t need = mla_plan_size_for_clusters(batch, s_q, h_q, num_clusters);
  if (need == 0) return MLA_ERR_INVALID_ARG;
  if (tile_meta_bytes < need) return MLA_ERR_WORKSPACE;
  plan_host(cache_seqlens_host, batch, s_q, h_q, num_clusters,
            static_cast<int32_t*>(tile_meta_host));
  return MLA_OK;
}

int mla_decode_plan(const int32_t* cache_seqlens, int batch, int s_q, int h_q, void* tile_meta,
                    size_t tile_meta_bytes, void* stream) {
  if (!cache_seqlens || !tile_meta || !shape_ok(batch, s_q, h_q) || !aligned(tile_meta, 8) ||
      !aligned(cache_seqlens, 4))
    return MLA_ERR_INVALID_ARG;
  int device = 0;
  if (cudaGetDevice(&device) != cudaSuccess) return MLA_ERR_CUDA;
  const int st = setup_device(device);
  if (st != MLA_OK) return st;
  const DeviceState& d = g_dev[device];
  const size_t need = mla_plan_size_for_clusters(batch, s_q, h_q, d.num_clusters);
  if (need == 0) return MLA_ERR_INVALID_ARG;
  if (tile_meta_bytes < need) return MLA_ERR_WORKSPACE;
  const size_t smem = batch <= kPlanSmemBatch
                          ? sizeof(int64_t) * (size_t)(batch + 1) + sizeof(int32_t) * (size_t)batch
                          : 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1);
  cfg.blockDim = dim3(kPlanThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, mla_plan_kernel, cache_seqlens, batch, s_q, h_q,
                            d.num_clusters, static_cast<int32_t*>(tile_meta), d.err) ==
                 cudaSuccess
             ? MLA_OK
             : MLA_ERR_CUDA;
}

}  // extern "C"

namespace {

// Shared checks of the decode entry points; fills the kernel parameters.
int prepare_decode(const void* q, const void* kv_cache, int num_pages, const int32_t* block_table,
                   int max_pages, const int32_t* cache_seqlens, int batch, int s_q, int h_q,
                   const void* tile_meta, void* out, float* lse, float softmax_scale,
                   void* workspace, size_t workspace_bytes, DecodeParams* p, int* num_clusters,
                   int* num_sms) {
  if (!q || !kv_cache || !block_table || !cache_seqlens || !tile_meta || !out || !lse)
    return MLA_ERR_INVALID_ARG;
  if (!shape_ok(batch, s_q, h_q) || num_pages < 1 || max_pages < 1 ||
      (int64_t)num_pages * kPageTokens >= ((int64_t)1 << 31) || !isfinite(softmax_scale))
    return MLA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(kv_cache, 16) || !aligned(out, 16) || !aligned(lse, 4) ||
      !aligned(block_table, 4) || !aligned(cache_seqlens, 4) || !aligned(tile_meta, 8))
    return MLA_ERR_INVALID_ARG;
  int device = 0;
  if (cudaGetDevice(&device) != cudaSuccess) return MLA_ERR_CUDA;
  const int st = setup_device(device);
  if (st != MLA_OK) return st;
  const DeviceState& d = g_dev[device];
  if (plan_group_clusters(d.num_clusters, plan_tiles(s_q, h_q)) < 1) return MLA_ERR_INVALID_ARG;
  const int64_t need = workspace_bytes_for(d.num_clusters);
  if (!workspace || (int64_t)workspace_bytes < need) return MLA_ERR_WORKSPACE;
  if (!aligned(workspace, 256)) return MLA_ERR_INVALID_ARG;
  p->q = q;
  p->kv = kv_cache;
  p->block_table = block_table;
  p->seqlens = cache_seqlens;
  p->indices = nullptr;
  p->cache_len = nullptr;
  p->topk = 0;
  p->plan = static_cast<const int32_t*>(tile_meta);
  p->out = out;
  p->out_v8 = (reinterpret_cast<uintptr_t>(out) & 31u) == 0 ? 1 : 0;
  p->lse = lse;
  p->out_f32 = 0;
  const int64_t slots = workspace_slots(d.num_clusters);
  p->ws_o = static_cast<float*>(workspace);
  p->ws_lse = static_cast<float*>(workspace) + slots * kSlotFloats;
  p->err = d.err;
  p->batch = batch;
  p->s_q = s_q;
  p->h_q = h_q;
  p->max_pages = max_pages;
  p->num_pages = num_pages;
  p->scale_log2 = softmax_scale * 1.4426950408889634f;
  *num_clusters = d.num_clusters;
  *num_sms = d.num_sms;
  return MLA_OK;
}

int attend(const void* q, const void* kv_cache, const DecodeParams& p, int num_clusters,
           cudaStream_t s) {
  TensorMaps maps;
  const uint64_t q_rows = (uint64_t)p.batch * p.s_q * p.h_q;
  const uint64_t kv_rows = (uint64_t)p.num_pages * kPageTokens;
  if (!make_map(&maps.q_rope, q, q_rows, 32, kTileRows, CU_TENSOR_MAP_SWIZZLE_64B) ||
      !make_map(&maps.kv_lat, kv_cache, kv_rows, 64, kPageTokens, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_map(&maps.kv_rope, kv_cache, kv_rows, 32, kPageTokens, CU_TENSOR_MAP_SWIZZLE_64B))
    return MLA_ERR_CUDA;
  return launch_decode(maps, p, num_clusters, s) == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}


// mla_decode and mla_decode_f32: the main kernel, then the combine; out_f32
// selects the output element type.
int decode_impl(const void* q, const void* kv_cache, int num_pages, const int32_t* block_table,
                int max_pages, const int32_t* cache_seqlens, int batch, int s_q, int h_q,
                const void* tile_meta, void* out, int out_f32, float* lse, float softmax_scale,
                void* workspace, size_t workspace_bytes, void* stream) {
  DecodeParams p;
  int nc = 0, sms = 0;
  const int rc = prepare_decode(q, kv_cache, num_pages, block_table, max_pages, cache_seqlens,
                                batch, s_q, h_q, tile_meta, out, lse, softmax_scale, workspace,
                                workspace_bytes, &p, &nc, &sms);
  if (rc != MLA_OK) return rc;
  p.out_f32 = out_f32;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int a = attend(q, kv_cache, p, nc, s);
  if (a != MLA_OK) return a;
  return launch_combine(p, nc, sms, s) == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

int sparse_impl(const void* q, const void* kv_cache, int num_pages, const int32_t* block_table,
                int max_pages, const int32_t* cache_seqlens, const int32_t* indices, int topk,
                const int32_t* counts, int batch, int h_q, const void* tile_meta, void* out,
                int out_f32, float* lse, float softmax_scale, void* workspace,
                size_t workspace_bytes, void* stream) {
  if (!indices || !counts || !cache_seqlens || topk < 1 || !aligned(indices, 4) ||
      !aligned(counts, 4) || (int64_t)batch * topk >= ((int64_t)1 << 31))
    return MLA_ERR_INVALID_ARG;
  DecodeParams p;
  int nc = 0, sms = 0;
  // the counts take the place of the sequence lengths: the plan splits them
  // into chunks of 64 listed positions, and the kernel masks past them
  const int rc = prepare_decode(q, kv_cache, num_pages, block_table, max_pages, counts, batch,
                                1, h_q, tile_meta, out, lse, softmax_scale, workspace,
                                workspace_bytes, &p, &nc, &sms);
  if (rc != MLA_OK) return rc;
  if (!aligned(cache_seqlens, 4)) return MLA_ERR_INVALID_ARG;
  p.indices = indices;
  p.cache_len = cache_seqlens;
  p.topk = topk;
  p.out_f32 = out_f32;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int a = attend(q, kv_cache, p, nc, s);
  if (a != MLA_OK) return a;
  return launch_combine(p, nc, sms, s) == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

}  // namespace

extern "C" {

int mla_decode_attend(const void* q, const void* kv_cache, int num_pages,
                      const int32_t* block_table, int max_pages, const int32_t* cache_seqlens,
                      int batch, int s_q, int h_q, const void* tile_meta, void* out, float* lse,
                      float softmax_scale, void* workspace, size_t workspace_bytes, void* stream) {
  DecodeParams p;
  int nc = 0, sms = 0;
  const int rc = prepare_decode(q, kv_cache, num_pages, block_table, max_pages, cache_seqlens,
                                batch, s_q, h_q, tile_meta, out, lse, softmax_scale, workspace,
                                workspace_bytes, &p, &nc, &sms);
  if (rc != MLA_OK) return rc;
  return attend(q, kv_cache, p, nc, static_cast<cudaStream_t>(stream));
}

int mla_decode_combine(int batch, int s_q, int h_q, const void* tile_meta, void* out, float* lse,
                       void* workspace, size_t workspace_bytes, void* stream) {
  if (!tile_meta || !out || !lse || !shape_ok(batch, s_q, h_q) || !aligned(tile_meta, 8) ||
      !aligned(out, 16) || !aligned(lse, 4))
    return MLA_ERR_INVALID_ARG;
  int device = 0;
  if (cudaGetDevice(&device) != cudaSuccess) return MLA_ERR_CUDA;
  const int st = setup_device(device);
  if (st != MLA_OK) return st;
  const DeviceState& d = g_dev[device];
  const int64_t need = workspace_bytes_for(d.num_clusters);
  if (!workspace || (int64_t)workspace_bytes < need) return MLA_ERR_WORKSPACE;
  if (!aligned(workspace, 256)) return MLA_ERR_INVALID_ARG;
  DecodeParams p = {};
  p.plan = static_cast<const int32_t*>(tile_meta);
  p.out = out;
  p.lse = lse;
  p.out_f32 = 0;
  const int64_t slots = workspace_slots(d.num_clusters);
  p.ws_o = static_cast<float*>(workspace);
  p.ws_lse = static_cast<float*>(workspace) + slots * kSlotFloats;
  p.err = d.err;
  p.batch = batch;
  p.s_q = s_q;
  p.h_q = h_q;
  return launch_combine(p, d.num_clusters, d.num_sms, static_cast<cudaStream_t>(stream)) ==
                 cudaSuccess
             ? MLA_OK
             : MLA_ERR_CUDA;
}

int mla_decode(const void* q, const void* kv_cache, int num_pages, const int32_t* block_table,
               int max_pages, const int32_t* cache_seqlens, int batch, int s_q, int h_q,
               const void* tile_meta, void* out, float* lse, float softmax_scale,
               void* workspace, size_t workspace_bytes, void* stream) {
  return decode_impl(q, kv_cache, num_pages, block_table, max_pages, cache_seqlens, batch, s_q,
                     h_q, tile_meta, out, 0, lse, softmax_scale, workspace, workspace_bytes,
                     stream);
}

int mla_decode_f32(const void* q, const void* kv_cache, int num_pages,
                   const int32_t* block_table, int max_pages, const int32_t* cache_seqlens,
                   int batch, int s_q, int h_q, const void* tile_meta, float* out, float* lse,
                   float softmax_scale, void* workspace, size_t workspace_bytes, void* stream) {
  return decode_impl(q, kv_cache, num_pages, block_table, max_pages, cache_seqlens, batch, s_q,
                     h_q, tile_meta, out, 1, lse, softmax_scale, workspace, workspace_bytes,
                     stream);
}

int mla_decode_sparse(const void* q, const void* kv_cache, int num_pages,
                      const int32_t* block_table, int max_pages, const int32_t* cache_seqlens,
                      const int32_t* indices, int topk, const int32_t* counts, int batch, int h_q,
                      const void* tile_meta, void* out, float* lse, float softmax_scale,
                      void* workspace, size_t workspace_bytes, void* stream) {
  return sparse_impl(q, kv_cache, num_pages, block_table, max_pages, cache_seqlens, indices, topk,
                     counts, batch, h_q, tile_meta, out, 0, lse, softmax_scale, workspace,
                     workspace_bytes, stream);
}

int mla_decode_sparse_f32(const void* q, const void* kv_cache, int num_pages,
                          const int32_t* block_table, int max_pages,
                          const int32_t* cache_seqlens, const int32_t* indices, int topk,
                          const int32_t* counts, int batch, int h_q, const void* tile_meta,
                          float* out, float* lse, float softmax_scale, void* workspace,
                          size_t workspace_bytes, void* stream) {
  return sparse_impl(q, kv_cache, num_pages, block_table, max_pages, cache_seqlens, indices, topk,
                     counts, batch, h_q, tile_meta, out, 1, lse, softmax_scale, workspace,
                     workspace_bytes, stream);
}

int mla_selftest_wait_timeout(void* stream) {
  int device = 0;
  if (cudaGetDevice(&device) != cudaSuccess) return MLA_ERR_CUDA;
  const int st = setup_device(device);
  if (st != MLA_OK) return st;
  return launch_wait_selftest(g_dev[device].err, static_cast<cudaStream_t>(stream)) ==
                 cudaSuccess
             ? MLA_OK
             : MLA_ERR_CUDA;
}

int mla_check_device_error(void* stream) {
  int device = 0;
  if (cudaGetDevice(&device) != cudaSuccess) return MLA_ERR_CUDA;
  const int st = setup_device(device);
  if (st != MLA_OK) return st;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return MLA_ERR_CUDA;
  int v = 0;
  if (cudaMemcpy(&v, g_dev[device].err, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess)
    return MLA_ERR_CUDA;
  if (v != 0) {
    const int zero = 0;
    if (cudaMemcpy(g_dev[device].err, &zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess)
      return MLA_ERR_CUDA;
  }
  return v;
}

const char* mla_strerror(int code) {
  switch (code) {
    case MLA_OK: return "ok";
    case MLA_ERR_INVALID_ARG: return "invalid argument (null pointer, misalignment or unsupported shape)";
    case MLA_ERR_WORKSPACE: return "plan or workspace buffer too small";
    case MLA_ERR_CUDA: return "CUDA runtime error";
    case MLA_ERR_DEVICE_TIMEOUT: return "a bounded device wait timed out";
    case MLA_ERR_DEVICE_BOUNDS: return "out-of-range page index or negative sequence length";
    case MLA_ERR_UNSUPPORTED_DEVICE: return "device is not sm_103 (GB300)";
    case MLA_ERR_PLAN: return "tile metadata does not match this call";
    default: return "unknown error";
  }
}

}  // extern "C"

namespace mla {
cudaError_t launch_combine(const DecodeParams& p, int /*num_clusters*/, int num_sms,
                           cudaStream_t stream) {
  const int tiles = plan_tiles(p.s_q, p.h_q);
  const int64_t jobs = (int64_t)p.batch * tiles * ((kDv / 4) / kCombineQuads);
  // four CTAs per SM only when three would need another wave
  const bool four = jobs > (int64_t)num_sms * 3;
  const int64_t cap = (int64_t)num_sms * (four ? 4 : 3);
  const int grid = (int)(jobs < cap ? jobs : cap);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kCombineWarps * 32);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return four ? cudaLaunchKernelEx(&cfg, mla_combine_kernel<4, 4>, p)
              : cudaLaunchKernelEx(&cfg, mla_combine_kernel<6, 3>, p);
}
}  // namespace mla
