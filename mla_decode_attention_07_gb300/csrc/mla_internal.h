// Internal interfaces between the translation units of libmla.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "mla_plan.h"

namespace mla {

constexpr int kDqk = 576;  // latent (512) + rotary (64) dims per cache row
constexpr int kDv = 512;   // value dims = the first 512 dims of the row

// Everything the decode kernel needs besides its four tensor maps.
struct DecodeParams {
  const void* q;      // bf16 [B, s_q, h_q, 576]
  const void* kv;     // bf16 [num_pages, 64, 1, 576]
  const int32_t* block_table;
  const int32_t* seqlens;      // keys per entry: cache lengths, or the sparse counts
  const int32_t* indices;      // sparse: [B, topk] token positions; null for dense
  const int32_t* cache_len;    // sparse: cache lengths (bounds of the positions)
  int topk;
  const int32_t* plan;
  void* out;          // [B, s_q, h_q, 512]: bf16, or fp32 when out_f32
  float* lse;         // fp32 [B, h_q, s_q]
  float* ws_o;        // fp32 [slots][512 / 4][128 rows][4]
  float* ws_lse;      // fp32 [slots, 128]
  int* err;           // device error word
  int batch, s_q, h_q, max_pages, num_pages;
  int out_f32;        // 1: out is fp32 (the normalised fp32 result, unrounded)
  int out_v8;         // 1: out is 32-byte aligned (row pieces go out as 32-byte stores)
  float scale_log2;   // softmax_scale * log2(e)
};

struct TensorMaps {
  CUtensorMap q_rope, kv_lat, kv_rope;
};

// Partial results: one slot holds 128 rows x 512 fp32 plus 128 lse values.
constexpr int64_t kSlotFloats = (int64_t)kTileRows * kDv;

// Upper bound on the split slots any plan for `num_clusters` clusters needs:
// every group of clusters has at most 2 * (clusters in group) split parts
// belonging to entries with two or more splits.
MLA_HD int64_t workspace_slots(int num_clusters) { return 2 * (int64_t)num_clusters; }

// Decode kernel (mla_decode_sm103.cu).
int decode_smem_bytes();
cudaError_t decode_kernel_setup(int device);
int decode_max_clusters(int device);  // co-resident 2-CTA clusters, or < 0
cudaError_t launch_wait_selftest(int* err, cudaStream_t stream);
cudaError_t launch_decode(const TensorMaps& maps, const DecodeParams& p, int num_clusters,
                          cudaStream_t stream);

// Decode kernel for at most 32 query rows per entry (mla_decode_narrow_sm103.cu):
// the same plan, partials and combine as the general kernel.  launch_decode
// routes dense calls to it when narrow_decode_shape holds.
bool narrow_decode_shape(int s_q, int h_q, int batch, int max_pages, int num_clusters);
cudaError_t narrow_kernel_setup();
int narrow_max_clusters();   // co-resident 2-CTA clusters, or < 0
cudaError_t launch_decode_narrow(const CUtensorMap& kv_map, const DecodeParams& p,
                                 int num_clusters, cudaStream_t stream);

// Device set-up shared by every entry point (mla_api.cu): the current device,
// its SM count and the address of its device error word; MLA_OK or an error.
int device_current(int* device, int* num_sms, int** err);

// cuTensorMapEncodeTiled through the runtime's driver entry point; `rank`
// dims (innermost first), rank - 1 byte strides, a box of `box` elements.
bool encode_tiled_map(CUtensorMap* m, CUtensorMapDataType dtype, int rank, const void* base,
                      const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box,
                      CUtensorMapSwizzle swz);

// Combine kernel (mla_api.cu).
cudaError_t launch_combine(const DecodeParams& p, int num_clusters, int num_sms,
                           cudaStream_t stream);

}  // namespace mla
