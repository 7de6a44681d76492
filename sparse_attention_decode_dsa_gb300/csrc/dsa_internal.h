// Internal declarations shared by the host API and the kernel translation units.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "../../include/dsa.h"

namespace dsa {

constexpr int kPage = 64;
constexpr int kMaxTopK = 2048;
constexpr int kMaxIdxHeads = 64;
constexpr int kMaxSfaHeads = 128;
constexpr int kLatentDim = 576;
constexpr int kValueDim = 512;
constexpr int kTopkBins = 4096;              // per-row histogram of the keys' top 12 bits
constexpr int kMaxVisible = 1 << 20;         // longest row (positions) the indexer handles

constexpr int kMaxDevices = 128;             // device ordinals the per-device caches cover

// Streaming multiprocessors of the current device (looked up once per device).  Launch
// plans, and so the attention's workspace size, depend on it.
int device_sm_count();
// The pipeline wait limit the tensor-core kernels use by default (cycles, about 2 s).
long long sm100_default_wait_limit();

// Fixed scratch of dsa_indexer_topk_noalloc (noalloc.cu): its size, and its device
// address on the current device, looked up once per device.  *ptr stays null (with
// cudaSuccess) for a device ordinal at or beyond kMaxDevices.
constexpr size_t kNoAllocScratchBytes = size_t(8) << 20;
cudaError_t noalloc_scratch(void** ptr, int* device);

// Everything a kernel needs to locate a token's row, sequence and visible range.
struct TokenView {
  const int32_t* token_seq;  // may be null: token i is batch row i
  const int32_t* token_pos;  // may be null: seq_len - 1
  const int32_t* seq_lens;
  const int32_t* block_table;
  int32_t batch, max_pages, num_pages, n_tokens;
  int32_t max_visible;       // host-planned bound on any token's visible count
};

// Score pass: one row per query token; scores[row * stride + t] for visible t.
struct ScoreParams {
  TokenView tv;
  const void* q;           // [T, H, d]
  const void* q_scale;     // null | f32 [T] | u8 [T, H, d/32]
  const float* head_w;     // [T, H]
  const void* k;           // [num_pages, 64, d]
  const void* k_scale;     // null | f32 [num_pages, 64] | u8 [num_pages, 64, d/32]
  float* scores;           // workspace
  uint32_t* hist;          // workspace [T, kTopkBins]: counts of the keys' top 12 bits (zeroed)
  int64_t score_stride;
  uint32_t* err;
  int32_t n_heads, dim, act, max_page_blocks;
  int32_t q_dep;           // 1: q is written by the preceding kernel (wait before reading it)
  const float* qt;         // q~ [T, dim] f32 (the folded-query kernel only)
  int32_t seg_rows;        // row-blocked kernel: rows per segment (consecutive rows of one
                           // sequence; n_tokens is a multiple of it)
  int64_t wait_limit;      // tensor-core kernel: cycles a pipeline wait may take before it
                           // gives up (DSA_DEVERR_TIMEOUT); the default unless a test lowers it
};

struct TopkParams {
  TokenView tv;
  const float* scores;
  const uint32_t* hist;
  int64_t score_stride;
  int32_t* out_idx;
  float* out_score;  // may be null
  uint32_t* err;
  int32_t top_k;
};

struct SfaParams {
  TokenView tv;
  const uint16_t* q;       // bf16 [T, H, 576]
  const uint16_t* kv;      // bf16 [num_pages, 64, 576] (bf16 cache)
  const uint8_t* kv_codes; // FP8 cache: e4m3 [num_pages, 64, 512]; null for a bf16 cache
  const float* kv_scale;   //   f32 [num_pages, 64, 4]: one scale per 128-dim tile
  const uint16_t* kv_rope; //   bf16 [num_pages, 64, 64]
  const int32_t* idx;      // [T, K]
  uint16_t* out;           // bf16 [T, H, 512]
  float* part_o;           // [T, S, 2 halves, 256 dims, HP]: each split's O / l (more than two
                           // splits); HP = H rounded up to a multiple of 4
  float* part_lse;         // [T, S, 2 halves, HP]: each split's log2-sum-exp of its logits
  uint32_t* err;
  int32_t n_heads, top_k, n_splits, split_len;
  int32_t sib_merge;       // two splits, merged inside a cluster of four (no partials in memory)
  float scale_log2;        // softmax_scale * log2(e)
};

// 2-D TMA map over `rows` rows of `row_elems` elements of `elem` bytes, 128-byte
// swizzle, box = 128 bytes x box_rows (tma_host.cu).
// `promote_l2`: let L2 fetch 256-byte blocks around each request (good for boxes of
// consecutive rows; for gathers of scattered rows it fetches bytes nobody asked for).
bool make_tma_2d_sw128(CUtensorMap* m, const void* base, uint64_t rows, int elem, int row_elems, int box_rows,
                       bool promote_l2 = true);
// Same with 64-byte swizzle and a 64-byte box inner extent, box_rows rows (no L2
// promotion); one-row boxes serve to gather 64-byte pieces of scattered rows.
bool make_tma_2d_sw64_rows(CUtensorMap* m, const void* base, uint64_t rows, int elem, int row_elems,
                           int box_rows = 1);

// cudaFuncSetAttribute(MaxDynamicSharedMemorySize) once per device and kernel (the
// attribute persists for the context; setting it on every launch costs host time on the
// launch path).  `done` is the kernel's own per-device flag array.
template <typename F>
cudaError_t set_smem_once(F* kernel, int bytes, std::atomic<int> (&done)[kMaxDevices]) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < kMaxDevices && done[dev].load(std::memory_order_acquire) == bytes) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && dev >= 0 && dev < kMaxDevices) done[dev].store(bytes, std::memory_order_release);
  return e;
}

// Launch with programmatic stream serialization: the kernel may start while the previous
// kernel in the stream is finishing; it calls pdl_wait() before touching what that
// kernel writes (or anything a later pass overwrites).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}
// Same, in thread-block clusters of `cluster_x` CTAs along x.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl_cluster(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                               unsigned cluster_x, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = cluster_x;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

// Launchers (each returns the cudaError_t of its launch).
cudaError_t launch_score(const ScoreParams& p, dsa_dtype_t dt, dsa_scale_t sk, cudaStream_t s);
bool score_tc_supported(dsa_dtype_t dt, int dim, int n_heads);
cudaError_t launch_score_tc(const ScoreParams& p, dsa_dtype_t dt, dsa_scale_t sk, cudaStream_t s);
bool score_stream_supported(dsa_act_t act, int dim);
// q~ scratch: [n_tokens, dim] f32 in the workspace
cudaError_t launch_score_stream(const ScoreParams& p, dsa_dtype_t dt, dsa_scale_t sk, float* qt, cudaStream_t s);
// q~ alone (f32 [n_tokens, dim], query scales folded in)
cudaError_t launch_qtilde(const ScoreParams& p, dsa_dtype_t dt, dsa_scale_t sk, float* qt, cudaStream_t s);
// e4m3 keys, identity activation, d = 128: the TMA page ring of the tensor-core kernel,
// each key's dot product with q~ (key scales applied) on the CUDA cores from shared memory
bool score_fold_supported(dsa_dtype_t dt, dsa_scale_t sk, dsa_act_t act, int dim);
cudaError_t launch_score_fold(const ScoreParams& p, dsa_scale_t sk, const float* qt, cudaStream_t s);
// bf16, identity activation: the head-collapsed query split into 3 bf16 terms, laid out
// as `stride` rows per token [n_tokens, stride, dim] (terms, then zero rows) with weights
// [n_tokens, stride] (1, 1, 1, 0, ...; skipped when ws is null).  The row-blocked kernel
// takes stride 3 (consecutive tokens' terms back to back).  The workspace reserves
// kSplitQueryHeads rows per token for it.
// The query may be bf16, or e4m3 with its scales (folded into the sum exactly).
constexpr int kSplitQueryHeads = 16;
cudaError_t launch_qsplit(const ScoreParams& p, dsa_dtype_t dt, dsa_scale_t sk, uint16_t* qs, float* ws, int stride,
                          cudaStream_t s);
// e4m3 keys of sequence b for the row-blocked kernel: its first npv pages dequantised to
// bf16 compact pages kb [npv, 64, dim] (MX group scales applied; per-token scales copied
// to ks [npv * 64]), and bt_out[b * max_pages + j] = j (-1 for an invalid page id).
cudaError_t launch_kdequant(const ScoreParams& p, dsa_scale_t sk, int b, int npv, uint16_t* kb, float* ks,
                            int32_t* bt_out, cudaStream_t s);
// The row-blocked tensor-core score kernel: the tokens come in segments of p.seg_rows
// consecutive rows of one sequence (host checked); blocks of up to kBlockRows rows of a
// segment share each K tile; p.q is the stride-3 split query; bf16 keys, times
// p.k_scale[key] when that is set.
constexpr int kBlockRows = 21;
constexpr int kBlockedMaxSeg = 1024;  // longest segment of several sequences' rows (rows per launch)
cudaError_t launch_score_tc_blocked(const ScoreParams& p, cudaStream_t s);
cudaError_t launch_topk(const TopkParams& p, int32_t max_visible, cudaStream_t s);
cudaError_t launch_sfa_tc(const SfaParams& p, cudaStream_t s);
// More than two splits: the merge of the attention kernel's partials into p.out.
cudaError_t launch_sfa_combine(const SfaParams& p, cudaStream_t s);
cudaError_t launch_clear(void* p, size_t bytes, cudaStream_t s);  // bytes: multiple of 16

// Index prolog: MXFP8 quantisation (groups of 32) of bf16 rows, written to row i of
// codes / scales, or (append) to the cache row of token i's (page, slot).
struct Mxfp8Params {
  const uint16_t* x;   // [n_rows, dim] bf16, 16-byte aligned
  int64_t n_rows;
  int32_t dim;         // a multiple of 32
  uint8_t* codes;      // [rows, dim] e4m3, 8-byte aligned
  uint8_t* scales;     // [rows, dim / 32] E8M0
  bool append;         // destination from (token_seq, token_pos) through the page table
  TokenView tv;        // (append only)
  uint32_t* err;       // (append only) device error word
};
cudaError_t launch_mxfp8_quant(const Mxfp8Params& p, cudaStream_t s);

// Append of each new token's latent row ([T, 576] bf16) to its (page, slot) of the
// latent cache: bf16 rows (data), or FP8 (codes [.., 512] e4m3, scales [.., 4] f32 per
// 128-dim tile, rope [.., 64] bf16).
struct LatentAppendParams {
  const uint16_t* x;   // [n_rows, 576] bf16, 16-byte aligned
  int64_t n_rows;
  uint16_t* data;      // bf16 cache
  uint8_t* codes;      // FP8 cache
  float* scales;
  uint16_t* rope;
  TokenView tv;
  uint32_t* err;
};
cudaError_t launch_latent_append(const LatentAppendParams& p, bool fp8, cudaStream_t s);

// Append of each new token's key ([T, dim] bf16) to a bf16 K-index cache or an e4m3 one
// with one f32 scale per token.
struct IndexAppendParams {
  const uint16_t* x;   // [n_rows, dim] bf16
  int64_t n_rows;
  void* data;          // [pages, 64, dim] bf16 or e4m3
  float* scales;       // [pages, 64] (e4m3)
  TokenView tv;
  uint32_t* err;
};
cudaError_t launch_index_append(const IndexAppendParams& p, int dim, bool fp8, cudaStream_t s);

}  // namespace dsa
