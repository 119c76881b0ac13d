/*
 * libmla — paged Multi-head Latent Attention (MLA) decode for NVIDIA GB300
 * (sm_103a), behind a plain C ABI.
 *
 * The operation.  DeepSeek-style MLA decode, the FlashMLA kernel that the
 * TileLang talk uses as its worked example ("Tile级原语与自动推理机制融合，
 * TileAI社区发起人深度剖析TileLang核心技术与优势", section 什么是「TileLang」:
 * the ~50-line MLA kernel and its accum_s -> scores_max reduce).  The pages
 * name the kernel but print no formula; the result computed here is
 * scaled-dot-product attention of every query row over the latent cache rows
 * it may see:
 *
 *   for batch b, query token i < s_q, head h:
 *     n        = cache_seqlens[b] - s_q + 1 + i   (bottom-right causal)
 *     k_t      = kv_cache[block_table[b][t/64]][t%64][0][0:576],  t < n
 *     s_t      = softmax_scale * <q[b][i][h][0:576], k_t>
 *     lse      = ln(sum_t exp(s_t))
 *     out[0:512] = sum_t exp(s_t - lse) * k_t[0:512]
 *
 * Dims 0..511 of a cache row are the latent part (also the values), dims
 * 512..575 the rotary part.  One latent head is shared by all query heads.
 * A row with no visible key gets out = 0 and lse = -inf.
 *
 * Layouts (all row-major, densely packed):
 *   q            bf16  [batch, s_q, h_q, 576]        device
 *   kv_cache     bf16  [num_pages, 64, 1, 576]       device
 *   block_table  int32 [batch, max_pages]            device
 *   cache_seqlens int32 [batch]                      device (host for the
 *                                                    _host planner variant)
 *   out          bf16  [batch, s_q, h_q, 512]        device
 *   lse          fp32  [batch, h_q, s_q]             device
 *
 * Arithmetic: bf16 inputs; q.k and P.V products accumulate in fp32 on the
 * tensor cores.  The 576-wide q.k of a row is summed in two halves on the
 * two SMs of a cluster; the half that crosses to the row's owner is rounded
 * to a 24-bit float (relative error <= 2^-16, within the fp32 accumulation's
 * own bound for those 288 products).  Probabilities enter P.V as bf16; out is
 * normalised by the sum of those bf16 probabilities and rounded to bf16 (or
 * returned as fp32 by the _f32 entry points); lse comes from the fp32 sums.
 *
 * Ownership: the caller owns every buffer; the library allocates nothing on
 * any call.  Asynchrony: every call that takes a stream only enqueues work on
 * it and returns; errors found on the host are returned before anything is
 * enqueued.  Device-side faults of the bounded kind (a wait that timed out,
 * an out-of-range page index) are recorded in a device word and reported by
 * mla_check_device_error.  There is no CPU fallback: on a device that is not
 * sm_103 every entry point that would launch returns MLA_ERR_UNSUPPORTED_DEVICE.
 *
 * Supported shapes: 1 <= h_q <= 128, 1 <= s_q <= 8 (s_q * h_q query rows per
 * batch entry, processed in tiles of 128 rows), batch >= 1, page size 64,
 * d_qk = 576, d_v = 512, num_pages * 64 < 2^31.  q and kv_cache must be 16-byte
 * aligned, out 16-byte aligned, lse 4-byte aligned.
 */
#ifndef LIBMLA_MLA_H_
#define LIBMLA_MLA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Return codes. */
#define MLA_OK 0
#define MLA_ERR_INVALID_ARG (-1)        /* null pointer, misalignment, bad shape */
#define MLA_ERR_WORKSPACE (-2)          /* plan or workspace buffer too small */
#define MLA_ERR_CUDA (-3)               /* a CUDA runtime call or launch failed */
#define MLA_ERR_DEVICE_TIMEOUT (-4)     /* a bounded device wait ran out */
#define MLA_ERR_DEVICE_BOUNDS (-5)      /* a block_table entry was out of range */
#define MLA_ERR_UNSUPPORTED_DEVICE (-6) /* the device is not sm_103 */
#define MLA_ERR_PLAN (-7)               /* tile_meta does not match the call */

/* Element types of mla_gemm's operands and result. */
#define MLA_DTYPE_F16 0
#define MLA_DTYPE_BF16 1
#define MLA_DTYPE_F32 2

/* Number of two-CTA clusters the decode kernel runs as a persistent grid on
 * `device` (the SM count halved, limited by cluster occupancy).  Returns a
 * negative code on error.
 * Defined by: no passage.  The pages size no grid; the persistent grid of
 * this library's design needs the count to size the plan. */
int mla_num_clusters(int device);

/* Which decode kernel mla_decode (and mla_decode_f32, mla_decode_attend)
 * runs for a call of this shape on `device`: 1 = the narrow kernel (at most
 * 32 query rows per entry, s_q * h_q <= 32, and a block table of more than 4
 * pages per cluster, batch * max_pages > 4 * mla_num_clusters), 0 = the
 * general kernel; a negative code on error.  Both take the same plan and
 * workspace and meet the same tolerances; this only names the kernel a
 * profile will show.
 * Defined by: no passage (a choice between two designs of this library). */
int mla_decode_kernel_kind(int batch, int s_q, int h_q, int max_pages, int device);

/* Bytes of tile metadata for a plan of this shape on `device` (0 on error).
 * The plan is the split-KV work partition: which pages of which batch entry
 * each cluster processes, and how many partial results each entry has.
 * Defined by: no passage.  A C ABI cannot infer buffer sizes, so the caller
 * asks before allocating tile_meta (the pages describe no interface). */
size_t mla_plan_size(int batch, int s_q, int h_q, int device);

/* The same size for an explicit cluster count (what mla_decode_plan_host
 * needs for `num_clusters`).  0 on error.  Defined by: no passage (as
 * mla_plan_size). */
size_t mla_plan_size_for_clusters(int batch, int s_q, int h_q, int num_clusters);

/* Bytes of scratch mla_decode needs for split partials (fp32 partial outputs
 * and their lse) with a plan of this shape on `device` (0 on error).  The
 * bound does not depend on sequence lengths.
 * Defined by: no passage.  The split-KV partials are this library's
 * intermediate; the caller owns their memory, so it must learn the size. */
size_t mla_workspace_size(int batch, int s_q, int h_q, int device);

/* Split-KV planner (one small kernel).  Reads cache_seqlens (device int32
 * [batch]) and writes the tile metadata to tile_meta (device, at least
 * mla_plan_size bytes, 8-byte aligned).  One plan serves every layer of a
 * decode step that shares the sequence lengths.  Negative lengths are
 * treated as 0 and flagged as MLA_ERR_DEVICE_BOUNDS.
 * Defined by: the TileLang talk (page and section named at the top of this
 * file) centres on the FlashMLA decode kernel but prints no interface.
 * FlashMLA's public usage has two calls, a metadata call made once per
 * decode step and the attention call made per layer; this is the first:
 * it returns the split-KV tile metadata for the sequence lengths.
 * Errors: MLA_ERR_INVALID_ARG (null, misaligned, bad shape), MLA_ERR_WORKSPACE
 * (tile_meta_bytes too small), MLA_ERR_UNSUPPORTED_DEVICE, MLA_ERR_CUDA
 * (launch failed); nothing is enqueued on an error. */
int mla_decode_plan(const int32_t* cache_seqlens, int batch, int s_q, int h_q,
                    void* tile_meta, size_t tile_meta_bytes, void* stream);

/* The same plan computed on the host from host sequence lengths, for
 * `num_clusters` clusters; writes tile_meta_host (host memory).  The device
 * planner produces bit-identical metadata for the same inputs.
 * Defined by: as mla_decode_plan; the host form lets a caller that already
 * holds the lengths on the host skip the planner launch. */
int mla_decode_plan_host(const int32_t* cache_seqlens_host, int batch, int s_q, int h_q,
                         int num_clusters, void* tile_meta_host, size_t tile_meta_bytes);

/* Decode attention.  Launches the main kernel (persistent, two-CTA clusters;
 * TMA page streaming, tcgen05 MMAs with TMEM accumulators, online softmax)
 * and the LSE-combine kernel on `stream`.  tile_meta must come from
 * mla_decode_plan (or the host variant, copied to the device) for the same
 * batch, s_q, h_q and sequence lengths, in a buffer of at least
 * mla_plan_size(batch, s_q, h_q, device) bytes (the kernel reads its cluster
 * entry at the position this shape gives before it checks the header).  workspace: device scratch of at
 * least mla_workspace_size bytes, 256-byte aligned; its contents on entry do
 * not matter.  softmax_scale multiplies q.k before the softmax.  out is
 * bf16, the fp32 result rounded to nearest even.
 * Defined by: the TileLang talk, section 什么是「TileLang」: the DeepSeek MLA
 * (FlashMLA) decode kernel, whose scores feed the accum_s -> scores_max row
 * max; the pipeline section of the same talk (copies in their own stage,
 * only Copy and GEMM truly asynchronous).  The formula it computes is the
 * one at the top of this file; the argument list (q, kv_cache, block_table,
 * cache_seqlens, tile_meta, out, lse, softmax_scale, stream) is FlashMLA's
 * attention call in C form, plus the sizes a C ABI cannot infer and the
 * caller-owned workspace.
 * Errors: MLA_ERR_INVALID_ARG, MLA_ERR_WORKSPACE, MLA_ERR_UNSUPPORTED_DEVICE,
 * MLA_ERR_CUDA are returned before anything is enqueued; faults found on the
 * device (MLA_ERR_DEVICE_TIMEOUT, MLA_ERR_DEVICE_BOUNDS, MLA_ERR_PLAN) are
 * reported by mla_check_device_error. */
int mla_decode(const void* q, const void* kv_cache, int num_pages, const int32_t* block_table,
               int max_pages, const int32_t* cache_seqlens, int batch, int s_q, int h_q,
               const void* tile_meta, void* out, float* lse, float softmax_scale,
               void* workspace, size_t workspace_bytes, void* stream);

/* mla_decode with an fp32 output: out is float [batch, s_q, h_q, 512]
 * (16-byte aligned), the normalised fp32 result before any rounding; the
 * bf16 out of mla_decode is exactly this value rounded to nearest even.
 * Meant for callers that combine results further (for example partial
 * results over a sequence split across devices) and for checking the
 * kernel's arithmetic apart from the output format: a bf16 value of
 * magnitude 4 or more can be up to 2^-6 from the nearest representable one.
 * Defined by: as mla_decode.  Errors: as mla_decode. */
int mla_decode_f32(const void* q, const void* kv_cache, int num_pages,
                   const int32_t* block_table, int max_pages, const int32_t* cache_seqlens,
                   int batch, int s_q, int h_q, const void* tile_meta, float* out, float* lse,
                   float softmax_scale, void* workspace, size_t workspace_bytes, void* stream);

/* The two halves of mla_decode, for callers that want to schedule (or time)
 * them apart: mla_decode_attend launches only the main kernel (rows of batch
 * entries with one split get their final out/lse; the others leave fp32
 * partials in workspace), mla_decode_combine only the LSE-combine kernel
 * that merges those partials into out/lse.  Same arguments and rules as
 * mla_decode; the combine must follow the attend on the same stream with
 * the same tile_meta and workspace.
 * Defined by: as mla_decode (the split-KV decode and the LSE combine are
 * its two kernels; the pages name neither). */
int mla_decode_attend(const void* q, const void* kv_cache, int num_pages,
                      const int32_t* block_table, int max_pages, const int32_t* cache_seqlens,
                      int batch, int s_q, int h_q, const void* tile_meta, void* out, float* lse,
                      float softmax_scale, void* workspace, size_t workspace_bytes, void* stream);
int mla_decode_combine(int batch, int s_q, int h_q, const void* tile_meta, void* out, float* lse,
                       void* workspace, size_t workspace_bytes, void* stream);

/* Sparse decode: one query token per batch entry (s_q = 1) attending to a
 * listed subset of its cache rows instead of all of them.  The FlagTree
 * talk write-up ("FlagTree: Triton-TLE 言語拡張、タイルIRバックエンド、
 * およびコンパイラ最適化手法", section 性能テスト) reports SparseMLA decode
 * at 128K context without a mechanism; this is DeepSeek's form of it:
 *
 *   keys of entry b: the cache rows at token positions indices[b][j],
 *   j < counts[b] (a list: a repeated position counts twice); each
 *   position t in [0, cache_seqlens[b]) sits at
 *   kv_cache[block_table[b][t/64]][t%64]
 *   out, lse: as mla_decode over those keys (no causal mask)
 *
 *   indices  int32 [batch, topk]  device, positions past counts[b] ignored
 *   counts   int32 [batch]        device, 0 <= counts[b] <= topk
 *   q        bf16 [batch, 1, h_q, 576]; out bf16 [batch, 1, h_q, 512];
 *   lse      fp32 [batch, h_q, 1]
 *
 * tile_meta comes from mla_decode_plan(counts, batch, 1, h_q, ...): the plan
 * splits each entry's list into chunks of 64 positions the way it splits a
 * sequence into pages.  The kernel gathers each chunk's rows with 16-byte
 * asynchronous copies (the rows are scattered, so there is no page to load
 * whole).  A position outside [0, cache_seqlens[b]), a block-table entry
 * outside the pool or counts[b] > topk is flagged as MLA_ERR_DEVICE_BOUNDS
 * and its row read as zeros.  Other rules as mla_decode.
 * Defined by: the FlagTree write-up, section 性能テスト (SparseMLA at 128K
 * context); the mechanism and interface are this library's reading. */
int mla_decode_sparse(const void* q, const void* kv_cache, int num_pages,
                      const int32_t* block_table, int max_pages, const int32_t* cache_seqlens,
                      const int32_t* indices, int topk, const int32_t* counts, int batch, int h_q,
                      const void* tile_meta, void* out, float* lse, float softmax_scale,
                      void* workspace, size_t workspace_bytes, void* stream);

/* mla_decode_sparse with an fp32 output (float [batch, 1, h_q, 512], 16-byte
 * aligned), as mla_decode_f32 is to mla_decode.  Defined by: as
 * mla_decode_sparse. */
int mla_decode_sparse_f32(const void* q, const void* kv_cache, int num_pages,
                          const int32_t* block_table, int max_pages,
                          const int32_t* cache_seqlens, const int32_t* indices, int topk,
                          const int32_t* counts, int batch, int h_q, const void* tile_meta,
                          float* out, float* lse, float softmax_scale, void* workspace,
                          size_t workspace_bytes, void* stream);

/* ---------------------------------------------------------------------
 * The steps before the decode call, and the tensor-core GEMM.
 * --------------------------------------------------------------------- */

/* Appends the new tokens' latent cache rows.  For batch entry b and new
 * token i < s_q, position t = cache_seqlens[b] - s_q + i (the lengths
 * already count the new tokens, as mla_decode expects), and
 *   kv_cache[block_table[b][t / 64]][t % 64][0][0:576] = kv_new[b][i][0:576]
 * bit for bit; nothing else in the cache changes.
 *   kv_new        bf16 [batch, s_q, 576]      device, 16-byte aligned
 *   kv_cache      bf16 [num_pages, 64, 1, 576] device, 16-byte aligned
 *   block_table   int32 [batch, max_pages]    device
 *   cache_seqlens int32 [batch]               device
 * A position below 0 or past the block table, or a page outside the pool,
 * is flagged as MLA_ERR_DEVICE_BOUNDS (read by mla_check_device_error) and
 * that row is skipped; the other rows are written.
 * Defined by: no passage.  The TileLang talk (section 什么是「TileLang」)
 * names the DeepSeek MLA decode kernel this feeds; the pages say nothing of
 * how the cache is filled, and this is DeepSeek's paged-cache write of the
 * 512 latent + 64 rotary dims of each new token.
 * Errors: MLA_ERR_INVALID_ARG (null, misaligned, bad size) before anything
 * is enqueued, MLA_ERR_UNSUPPORTED_DEVICE, MLA_ERR_CUDA. */
int mla_cache_append(const void* kv_new, void* kv_cache, int num_pages,
                     const int32_t* block_table, int max_pages, const int32_t* cache_seqlens,
                     int batch, int s_q, void* stream);

/* Query absorption: builds mla_decode's query from the per-head query parts.
 *   q[b][i][h][0:512]   = sum_{d<128} q_nope[b][i][h][d] * w_uk[h][d][0:512]
 *   q[b][i][h][512:576] = q_rope[b][i][h][0:64]
 *   q_nope bf16 [batch, s_q, h_q, 128], q_rope bf16 [batch, s_q, h_q, 64],
 *   w_uk bf16 [h_q, 128, 512] (the key up-projection of each head),
 *   q bf16 [batch, s_q, h_q, 576]; all device, 16-byte aligned.
 * The contraction runs on the tensor cores, per head and taken transposed
 * (latent dims x query rows; fp32 accumulation; q_latent rounded to bf16,
 * nearest even).
 * Defined by: no passage (as mla_cache_append): DeepSeek MLA's absorbed
 * form, in which W_UK is folded into the query so that the scores are taken
 * against the 512-dim latent cache directly.
 * Errors: MLA_ERR_INVALID_ARG before anything is enqueued,
 * MLA_ERR_UNSUPPORTED_DEVICE, MLA_ERR_CUDA; a bounded device wait that ran
 * out is reported by mla_check_device_error. */
int mla_q_absorb(const void* q_nope, const void* q_rope, const void* w_uk, void* q, int batch,
                 int s_q, int h_q, void* stream);

/* Tensor-core GEMM: C = A B with A [M, K] and B [K, N] row-major, both
 * in_dtype (MLA_DTYPE_F16 or MLA_DTYPE_BF16), fp32 accumulation, C [M, N]
 * row-major in out_dtype (F16, BF16: round to nearest even; or F32).
 * N and K must be multiples of 8; A, B, C 16-byte aligned; any M.
 * Defined by: the GEMM tutorial summary ("Designing high-performance GPU
 * kernels with TileLang: Tensor-Core GEMM", the comparison table): an FP16
 * 2048 x 2048 x 2048 GEMM measured against cuBLAS, relative error < 2e-2.
 * Errors: MLA_ERR_INVALID_ARG before anything is enqueued,
 * MLA_ERR_UNSUPPORTED_DEVICE, MLA_ERR_CUDA; a bounded device wait that ran
 * out is reported by mla_check_device_error. */
int mla_gemm(const void* A, const void* B, void* C, int M, int N, int K, int in_dtype,
             int out_dtype, void* stream);

/* Dense attention forward (FlashAttention style):
 *   for batch b, head h, query i < seqlen, keys t < seqlen (t <= i if causal):
 *     s_t = softmax_scale * q[b][i][h][0:d_qk] . k[b][t][h][0:d_qk]
 *     out[b][i][h][0:d_v] = sum_t softmax(s)_t v[b][t][h][0:d_v]   (bf16)
 *     lse[b][h][i] = ln sum_t exp(s_t)                             (fp32)
 *   q, k bf16 [batch, seqlen, heads, d_qk]; v bf16 [batch, seqlen, heads,
 *   d_v]; out bf16 [batch, seqlen, heads, d_v]; all device, 16-byte aligned;
 *   lse fp32 [batch, heads, seqlen], 4-byte aligned.
 * Supported: d_qk in {64, 128, 192}, d_v = 128, softmax_scale > 0.  MLA
 * prefill in DeepSeek's MHA form is d_qk = 192 (128 + 64 rotary), d_v = 128,
 * causal, 128 heads.  bf16 inputs, fp32 accumulation on the tensor cores,
 * probabilities enter P.V as bf16; out is normalised by their sum.
 * Defined by: the TileLang talk, performance section (MLA, FlashAttention
 * and block-sparse kernels on par with CUTLASS), and the GEMM tutorial
 * summary, key capabilities (FlashAttention; GEMM + softmax fused so the
 * scores stay out of HBM); neither prints the formula, which is the plain
 * definition above.
 * Errors: MLA_ERR_INVALID_ARG before anything is enqueued,
 * MLA_ERR_UNSUPPORTED_DEVICE, MLA_ERR_CUDA; a bounded device wait that ran
 * out is reported by mla_check_device_error. */
int mla_attention_fwd(const void* q, const void* k, const void* v, void* out, float* lse,
                      int batch, int seqlen, int heads, int d_qk, int d_v, int causal,
                      float softmax_scale, void* stream);

/* Failure-path self-test: enqueues a two-CTA kernel whose only wait, on a
 * barrier nothing completes, runs through the same bounded wait as the
 * decode kernel.  After about 2 s it gives up, records
 * MLA_ERR_DEVICE_TIMEOUT (read and cleared by mla_check_device_error) and
 * returns; the context stays usable.  For tests of the failure path only.
 * Defined by: no passage; the pages describe no failure handling. */
int mla_selftest_wait_timeout(void* stream);

/* mla_decode for callers that cannot allocate device memory: the same
 * arguments minus the workspace.  The paper has no counterpart; this entry
 * point exists for host frameworks whose allocator owns all device memory
 * (operators there may not call cudaMalloc) and for serving loops that must
 * never enter the CUDA allocator.  The split partials go to a static device
 * array inside the library, 38.1 MiB, enough for a plan on up to 76 two-CTA
 * clusters (a 152-SM GB300); a device needing more returns
 * MLA_ERR_WORKSPACE before anything is enqueued.  Every GPU that loads the
 * library keeps that array until the process exits.  All calls share it and
 * it keeps the last call's contents (nothing in it needs to start at zero),
 * so calls that overlap on the GPU race: serialise them.  The first call on
 * a device looks up the array's address with that device current; make it
 * before any stream capture.  Allocates nothing. */
int mla_decode_noalloc(const void* q, const void* kv_cache, int num_pages,
                       const int32_t* block_table, int max_pages, const int32_t* cache_seqlens,
                       int batch, int s_q, int h_q, const void* tile_meta, void* out, float* lse,
                       float softmax_scale, void* stream);

/* Synchronises `stream`, then returns and clears the device error word:
 * MLA_OK, MLA_ERR_DEVICE_TIMEOUT, MLA_ERR_DEVICE_BOUNDS or MLA_ERR_PLAN
 * (or MLA_ERR_CUDA if the synchronisation itself failed).
 * Defined by: no passage.  The launching calls only enqueue work, so errors
 * the kernels find (bounded waits that ran out, out-of-range page indices,
 * a plan that does not match the call) are collected in one device word
 * and read here; no device code traps. */
int mla_check_device_error(void* stream);

/* Static description of a return code (never null).  Defined by: no
 * passage; the C counterpart of an exception message. */
const char* mla_strerror(int code);

#ifdef __cplusplus
}
#endif

#endif /* LIBMLA_MLA_H_ */
