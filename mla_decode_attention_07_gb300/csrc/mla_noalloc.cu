// mla_decode_noalloc: paged MLA decode for callers that cannot allocate
// device memory.
//
// mla_decode needs a caller-provided workspace for the split-KV partials.
// Some callers cannot provide one: host frameworks and plugin hosts that own
// every byte of device memory through their own allocator and do not let an
// operator call cudaMalloc, and latency-critical serving loops that must never
// enter the CUDA allocator (cudaMalloc and cudaFree can synchronise the whole
// device).  For them this file keeps the scratch in a fixed, file-scope
// device array that the library itself owns; the caller passes only inputs,
// outputs and the plan.
//
// Limits and sharing:
//  * The array holds kStaticScratchBytes (38.1 MiB): the partial slots of a
//    plan for up to kStaticMaxClusters two-CTA clusters (76, i.e. a 152-SM
//    GB300).  A device that needs more (more clusters) is rejected with
//    MLA_ERR_WORKSPACE before anything is enqueued.  Every GPU that loads the
//    library holds the array until the process exits.
//  * All calls share the one array and it keeps whatever the last call left.
//    Nothing in it has to start at zero: every partial slot a call reads is
//    written earlier in that same call.  Calls that overlap on the GPU (on two
//    streams, or two host threads) race on the array and give wrong results;
//    serialise them.
//  * The first call on a device looks up the array's device address
//    (cudaGetSymbolAddress, with that device current); make that first call
//    before any stream capture.  Nothing here calls cudaMalloc, cudaFree or
//    any other allocating routine.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "mla.h"
#include "mla_internal.h"

namespace mla {
namespace {

constexpr int kStaticMaxClusters = 76;
constexpr size_t kStaticScratchBytes =
    (size_t)(2 * kStaticMaxClusters) * ((size_t)kSlotFloats * 4 + (size_t)kTileRows * 4);
constexpr int kMaxNoallocDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kStaticScratchBytes];

struct ScratchAddr {
  std::once_flag once;
  cudaError_t status = cudaErrorUnknown;
  void* ptr = nullptr;
};
ScratchAddr g_scratch_addr[kMaxNoallocDevices];

}  // namespace
}  // namespace mla

using namespace mla;

extern "C" int mla_decode_noalloc(const void* q, const void* kv_cache, int num_pages,
                                  const int32_t* block_table, int max_pages,
                                  const int32_t* cache_seqlens, int batch, int s_q, int h_q,
                                  const void* tile_meta, void* out, float* lse,
                                  float softmax_scale, void* stream) {
  int device = 0;
  if (cudaGetDevice(&device) != cudaSuccess) return MLA_ERR_CUDA;
  // the same code every other entry point gives for a device index it cannot track
  if (device < 0 || device >= kMaxNoallocDevices) return MLA_ERR_INVALID_ARG;
  ScratchAddr& s = g_scratch_addr[device];
  // One-time set-up on this device (it is the current one): the array's
  // device address.  Host code must not hand the symbol itself to a kernel.
  std::call_once(s.once, [&]() {
    void* p = nullptr;
    s.status = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    s.ptr = (s.status == cudaSuccess) ? p : nullptr;
  });
  if (s.status != cudaSuccess || s.ptr == nullptr) return MLA_ERR_CUDA;
  const size_t need = mla_workspace_size(batch, s_q, h_q, device);
  if (need == 0) {
    const int nc = mla_num_clusters(device);
    return nc < 0 ? nc : MLA_ERR_INVALID_ARG;
  }
  if (need > kStaticScratchBytes) return MLA_ERR_WORKSPACE;
  return mla_decode(q, kv_cache, num_pages, block_table, max_pages, cache_seqlens, batch, s_q,
                    h_q, tile_meta, out, lse, softmax_scale, s.ptr, kStaticScratchBytes, stream);
}
