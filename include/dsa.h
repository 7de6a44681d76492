/*
 * dsa.h -- C ABI of the GB300 DSA hot path: the fused Lightning Indexer (relevance
 * scoring, head weighting, head sum, Top-K) and Sparse Flash Attention over a paged
 * MLA latent cache.
 *
 * What the operations are (the pages this library follows):
 *   - "Adapting and Optimizing Inference for a New Model Architecture on Ascend",
 *     section 3.1: the indexer computes relevance scores of the query against a paged
 *     K cache, weights them per head and keeps the Top-K positions, in one fused unit
 *     that reads the paged cache directly and materialises no intermediate tensor; the
 *     sparse attention then reads only the selected KV entries.
 *   - "Day0 Inference Optimization on Ascend CANN", section 2 ("Deep Fusion of LI and
 *     SFA"): both operators run in BF16 and quantised modes, in prefill and decode;
 *     section 3: the indexer Q/K use MXFP8 with one scale per 32 elements.
 *   - "Inference Acceleration for Next-Gen Attention Architectures", section 3.2: the
 *     sparse attention reads non-contiguous positions through paged addressing.
 *
 * Conventions for every entry point:
 *   - Ownership: the caller allocates and owns every buffer, including the workspace.
 *     The library allocates no memory, keeps no state between calls (apart from
 *     per-device caches of the SM count and of the fixed scratch's address, the fixed
 *     scratch of dsa_indexer_topk_noalloc itself, and the test hook
 *     dsa_set_indexer_wait_limit: see those entry points) and may be called concurrently
 *     on different streams with different workspaces.
 *   - Workspace sizes depend on the arguments and on the current device (the attention
 *     splits its work by the device's SM count): size a workspace with the current
 *     device set to the one it will be used on.
 *   - Pointers marked "device" must be device (or managed) memory of the current CUDA
 *     device; "host" pointers are read synchronously during the call.  The index and
 *     latent caches, their scales, the attention query and its output must start on a
 *     16-byte boundary (they are moved in 16-byte or larger units); otherwise the call
 *     returns DSA_ERR_INVALID_ARG.
 *   - Execution: kernels are enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *     stream).  Argument checks run on the host before any launch; a failed check
 *     returns an error status and enqueues nothing.
 *   - Errors: status codes only, never C++ exceptions.  dsa_last_error_message() gives a
 *     human-readable reason for the most recent failure on the calling thread.
 *     Problems only the device can see (a page id outside the cache, a length beyond
 *     the page table) set bits of a 32-bit error word kept at the start of the
 *     workspace; the offending elements are treated as masked and no kernel traps.
 *     Read it with dsa_read_device_error().
 *   - Layouts are dense, row-major, with the last index fastest.  bf16 is IEEE
 *     bfloat16; e4m3 is OCP FP8 E4M3 (the "fn" variant: no infinities); E8M0 is an
 *     unsigned power-of-two exponent byte 2^(e-127).
 *   - Page size is 64 tokens.  Logical token t of batch row b lives in physical page
 *     block_table[b * max_pages_per_seq + t / 64], slot t % 64.
 */
#ifndef DSA_GB300_DSA_H
#define DSA_GB300_DSA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define DSA_ABI_VERSION 3

/* A cudaStream_t, kept opaque so that this header needs no CUDA header. */
typedef struct CUstream_st* dsa_stream_t;
/* A cudaEvent_t, kept opaque likewise. */
typedef struct CUevent_st* dsa_event_t;

typedef enum {
  DSA_OK = 0,
  DSA_ERR_INVALID_ARG = 1,  /* a NULL pointer, a negative size, inconsistent shapes  */
  DSA_ERR_UNSUPPORTED = 2,  /* a valid combination this build does not implement     */
  DSA_ERR_WORKSPACE = 3,    /* workspace NULL, too small or not 256-byte aligned     */
  DSA_ERR_CUDA = 4          /* a CUDA runtime call failed (launch, attribute, ...)   */
} dsa_status_t;

typedef enum { DSA_BF16 = 0, DSA_E4M3 = 1 } dsa_dtype_t;

typedef enum {
  DSA_SCALE_NONE = 0,          /* values are used as stored                              */
  DSA_SCALE_PER_TOKEN_F32 = 1, /* one f32 per token (all heads / dims share it)          */
  DSA_SCALE_MX_E8M0_G32 = 2    /* one E8M0 byte per 32 consecutive elements of a row     */
} dsa_scale_t;

/* Per-head activation applied to q_h . k_t before weighting.  The pages weight the raw
 * per-head scores (identity); RELU is offered for models that clamp them. */
typedef enum { DSA_ACT_IDENTITY = 0, DSA_ACT_RELU = 1 } dsa_act_t;

/* Device-side error bits (OR-ed into the workspace's error word). */
#define DSA_DEVERR_PAGE_ID 0x1u   /* a block_table entry outside [0, num_pages)          */
#define DSA_DEVERR_SEQ_LEN 0x2u   /* a seq_len outside [0, max_pages_per_seq * 64]        */
#define DSA_DEVERR_INDEX 0x4u     /* an SFA index outside [-1, visible count of its token]*/
#define DSA_DEVERR_TOKEN 0x8u     /* token_seq outside [0, batch) or token_pos < -1       */
#define DSA_DEVERR_TIMEOUT 0x10u  /* an internal pipeline wait gave up (~2 s); the kernel
                                     unwound without finishing its work                  */

/* Paged-cache addressing shared by the K-index cache and the latent cache. */
typedef struct {
  const int32_t* block_table;  /* device [batch, max_pages_per_seq]; entries past a
                                  sequence's last page are never read                  */
  const int32_t* seq_lens;     /* device [batch]: tokens stored for each batch row      */
  const int32_t* seq_lens_host;/* host [batch]: the same lengths, used to plan launches
                                  without a device->host copy                          */
  int32_t batch;               /* B >= 1                                               */
  int32_t max_pages_per_seq;   /* row stride of block_table, >= 1                      */
  int32_t page_size;           /* must be 64                                           */
  int32_t num_pages;           /* physical pages in each cache                         */
} dsa_page_table_t;

/* Query tokens.  Token i belongs to batch row token_seq[i] and sits at position
 * token_pos[i]; it may select positions t with t <= token_pos[i] and t < seq_len. */
typedef struct {
  int32_t n_tokens;               /* T >= 1                                             */
  const int32_t* token_seq;       /* device [T], or NULL: token i is batch row i (T == B) */
  const int32_t* token_pos;       /* device [T], or NULL: seq_len - 1 (decode)          */
  const int32_t* token_seq_host;  /* host [T]; required iff token_seq != NULL           */
  const int32_t* token_pos_host;  /* host [T]; required iff token_pos != NULL           */
} dsa_tokens_t;

/* K-index cache: one d-dim key per token, shared by all indexer heads. */
typedef struct {
  const void* data;        /* device [num_pages, 64, dim], bf16 or e4m3               */
  const void* scale;       /* device: NULL (SCALE_NONE) | f32 [num_pages, 64]
                              (PER_TOKEN_F32) | u8 E8M0 [num_pages, 64, dim/32] (MX)  */
  dsa_dtype_t dtype;       /* bf16 needs SCALE_NONE; e4m3 needs PER_TOKEN_F32 or MX   */
  dsa_scale_t scale_kind;
  int32_t dim;             /* d: 64 or 128                                            */
} dsa_index_cache_t;

/* Indexer query side. */
typedef struct {
  const void* q;           /* device [T, n_heads, dim], same dtype as the cache        */
  const void* q_scale;     /* device: NULL | f32 [T] | u8 E8M0 [T, n_heads, dim/32]    */
  dsa_dtype_t q_dtype;     /* must equal the cache dtype                              */
  dsa_scale_t q_scale_kind;/* must equal the cache scale kind                         */
  const float* head_w;     /* device [T, n_heads]: per-head weights                   */
  int32_t n_heads;         /* H_I: 1..64                                              */
  int32_t top_k;           /* K: 1..2048                                              */
  dsa_act_t act;
} dsa_indexer_args_t;

/* MLA latent cache: row = [latent (v_dim) | rope (dim - v_dim)].
 * bf16 (dtype DSA_BF16): data = bf16 [num_pages, 64, dim]; scale and rope NULL.
 * FP8 (dtype DSA_E4M3): the latent dims quantised per token in tiles of 128 ("Day0
 * Inference Optimization on Ascend CANN", section 3, "FP8 Block Quantization for SFA KV
 * Cache": tile 128, half the bytes read): data = e4m3 codes [num_pages, 64, v_dim],
 * scale = f32 [num_pages, 64, v_dim / 128] (latent element j of a row is
 * code * scale[j / 128]), rope = the rope dims in bf16 [num_pages, 64, dim - v_dim]
 * (the pages leave their storage open).  ABI version 3 added dtype, scale and rope;
 * zero them for a bf16 cache. */
typedef struct {
  const void* data;        /* device, see above                                       */
  int32_t dim;             /* 576                                                      */
  int32_t v_dim;           /* 512: the value is the leading v_dim entries of the row  */
  dsa_dtype_t dtype;       /* DSA_BF16 or DSA_E4M3                                    */
  const void* scale;       /* device f32 [num_pages, 64, v_dim / 128] (FP8), or NULL  */
  const void* rope;        /* device bf16 [num_pages, 64, dim - v_dim] (FP8), or NULL */
} dsa_latent_cache_t;

/* Sparse-attention query side. */
typedef struct {
  const void* q;           /* device [T, n_heads, dim] bf16                           */
  int32_t n_heads;         /* H: 1..128                                               */
  float softmax_scale;     /* logits = softmax_scale * q . row, e.g. 1/sqrt(576)      */
} dsa_sfa_args_t;

/* Optional per-launch timing: when passed, each kernel the call launches is bracketed
 * by a pair of caller-created events recorded on `stream`. */
#define DSA_TRACE_MAX 8
typedef struct {
  dsa_event_t begin[DSA_TRACE_MAX]; /* caller-created events (cudaEventCreate)         */
  dsa_event_t end[DSA_TRACE_MAX];
  int32_t n_recorded;               /* out: launches recorded                         */
  const char* name[DSA_TRACE_MAX];  /* out: static kernel names, in launch order      */
} dsa_trace_t;

/* ---- Lightning Indexer ---------------------------------------------------------- */
/* Bytes of workspace dsa_indexer_topk needs for these arguments (0 on bad arguments). */
size_t dsa_indexer_workspace_size(const dsa_indexer_args_t* args,
                                  const dsa_index_cache_t* cache,
                                  const dsa_page_table_t* pages,
                                  const dsa_tokens_t* tokens);

/* For every query token i: score I[t] = sum_h w[i,h] * act(q_i,h . k_t) (each side's
 * scales applied) over the visible positions t, then the top_k largest, ties to the
 * lower position.  out_idx (device int32 [T, top_k]) receives the chosen positions in
 * ascending order, padded with -1 when fewer than top_k are visible.  out_score
 * (device f32 [T, top_k], may be NULL) receives I[t] of each chosen position and NaN
 * in padded slots.  ws must be 256-byte aligned. */
dsa_status_t dsa_indexer_topk(const dsa_indexer_args_t* args,
                              const dsa_index_cache_t* cache,
                              const dsa_page_table_t* pages,
                              const dsa_tokens_t* tokens,
                              int32_t* out_idx, float* out_score,
                              void* ws, size_t ws_bytes,
                              dsa_stream_t stream, dsa_trace_t* trace);

/* ---- Sparse Flash Attention ----------------------------------------------------- */
size_t dsa_sparse_attn_workspace_size(const dsa_sfa_args_t* args,
                                      const dsa_page_table_t* pages,
                                      const dsa_tokens_t* tokens, int32_t top_k);

/* For every query token i and head h: out[i,h,:] = sum_j p_j row_j[:v_dim] with
 * p = softmax_j(softmax_scale * q[i,h,:] . row_j) over the rows of the positions
 * idx[i, 0..top_k) that are >= 0 (in any order; -1 entries are skipped).  A token with
 * no selected position gets out = 0.  out: device bf16 [T, n_heads, v_dim], rounded to
 * nearest even from f32. */
dsa_status_t dsa_sparse_attn(const dsa_sfa_args_t* args,
                             const dsa_latent_cache_t* cache,
                             const dsa_page_table_t* pages,
                             const dsa_tokens_t* tokens,
                             const int32_t* idx, int32_t top_k,
                             void* out, void* ws, size_t ws_bytes,
                             dsa_stream_t stream, dsa_trace_t* trace);

/* ---- The whole DSA step: indexer then sparse attention -------------------------- */
size_t dsa_fused_workspace_size(const dsa_indexer_args_t* iargs,
                                const dsa_index_cache_t* icache,
                                const dsa_sfa_args_t* sargs,
                                const dsa_page_table_t* pages,
                                const dsa_tokens_t* tokens);

/* dsa_indexer_topk followed by dsa_sparse_attn on its indices, stream-ordered, with no
 * host synchronisation.  out_idx (device int32 [T, top_k]) receives the indices; out is
 * the attention output as in dsa_sparse_attn. */
dsa_status_t dsa_fused_decode(const dsa_indexer_args_t* iargs,
                              const dsa_index_cache_t* icache,
                              const dsa_sfa_args_t* sargs,
                              const dsa_latent_cache_t* lcache,
                              const dsa_page_table_t* pages,
                              const dsa_tokens_t* tokens,
                              int32_t* out_idx, void* out,
                              void* ws, size_t ws_bytes,
                              dsa_stream_t stream, dsa_trace_t* trace);

/* ---- Lightning Indexer without a caller workspace ------------------------------ */
/* No counterpart in the pages: an entry point for callers that cannot allocate device
 * memory -- plugin hosts or serving runtimes that hand this library no allocator and
 * fix their memory budget up front, or request paths that must not call cudaMalloc
 * (it can synchronise the device).  Same inputs, outputs and semantics as
 * dsa_indexer_topk, but its scratch (the error word, key histograms and f32 score rows)
 * lives in a fixed 8 MiB array inside the library, one per device, held until the
 * process exits from the time the library's module holding it is loaded on that device
 * (under lazy module loading, the CUDA default: this entry point's first call there;
 * with CUDA_MODULE_LOADING=EAGER: context creation).  It allocates nothing.
 *   - Limit: 256 + n_tokens * (ceil(max visible / 64) * 64 * 4 + 16384 + 32 * dim + 64) bytes
 *     (each part rounded up to 256) must fit in 8 MiB (e.g. 32 decode tokens over 32768
 *     positions, or 8 over 131072); larger requests return DSA_ERR_WORKSPACE before any
 *     launch.
 *   - The first call on a device looks up the array's device address (set-up, once per
 *     device, under a lock); make that first call before any stream capture.
 *   - Every call on a device shares the one array and it keeps the last call's
 *     contents; what must start at zero (the key histograms) is cleared on `stream` by
 *     each call.  Calls that overlap on the GPU (different streams, or concurrent
 *     threads) race on it: order them on one stream.  Device-side error bits are not
 *     reported back (the error word there is never read or cleared); use
 *     dsa_indexer_topk with a workspace to read them. */
dsa_status_t dsa_indexer_topk_noalloc(const dsa_indexer_args_t* args,
                                      const dsa_index_cache_t* cache,
                                      const dsa_page_table_t* pages,
                                      const dsa_tokens_t* tokens,
                                      int32_t* out_idx, float* out_score,
                                      dsa_stream_t stream);

/* ---- Index prolog without weights: dynamic MXFP8 quantisation ------------------- */
/* MXFP8 with groups of 32 ("Day0 Inference Optimization on Ascend CANN", section 3,
 * "Full Quantization of LI with MXFP8"; "Adapting and Optimizing Inference for a New
 * Model Architecture on Ascend", section 4.2).  The pages leave the scale rule open; the
 * library takes the OCP microscaling one: each group of 32 consecutive elements of a
 * row shares the E8M0 scale 2^e with e = floor(log2(amax)) - 8 (amax: the group's
 * largest magnitude), clamped to [-127, 127], and e = -127 for an all-zero group; each
 * element is stored as the E4M3 value nearest x / 2^e, ties to even, saturating at
 * +-448.  Inputs must be finite.  The result is the layout the indexer reads with
 * DSA_SCALE_MX_E8M0_G32. */

/* Quantises n_rows rows of dim bf16 values, device x [n_rows, dim] (16-byte aligned;
 * dim a multiple of 32, at most 8192), into device codes e4m3 [n_rows, dim] (8-byte
 * aligned) and device scales E8M0 [n_rows, dim / 32]: e.g. the indexer query viewed as
 * [T * n_heads, dim].  n_rows == 0 enqueues nothing.  The caller owns every buffer. */
dsa_status_t dsa_quantize_mxfp8(const void* x, int64_t n_rows, int32_t dim,
                                void* codes, void* scales, dsa_stream_t stream);

/* Appends new keys to the paged MXFP8 K-index cache: the bf16 key of every token i,
 * device k_new [T, dim] (16-byte aligned), is quantised as above and written to the
 * cache row of token i's position: page block_table[b * max_pages_per_seq + pos / 64],
 * slot pos % 64, in cache_codes (device e4m3 [num_pages, 64, dim], 16-byte aligned) and
 * cache_scales (device E8M0 [num_pages, 64, dim / 32]).  b = token_seq[i] (or i) and
 * pos = token_pos[i], or seq_lens[b] - 1 when token_pos is NULL (the newest stored
 * position).  dim: 64 or 128 (the indexer's).  A position outside the page table sets
 * DSA_DEVERR_TOKEN, a page id outside [0, num_pages) DSA_DEVERR_PAGE_ID, in ws's error
 * word; that token is skipped and the others are written.  ws: 256-byte aligned, at
 * least 256 bytes (only the error word is used; it is not cleared by the call). */
dsa_status_t dsa_index_cache_append_mxfp8(const void* k_new, int32_t dim,
                                          const dsa_page_table_t* pages,
                                          const dsa_tokens_t* tokens,
                                          void* cache_codes, void* cache_scales,
                                          void* ws, size_t ws_bytes, dsa_stream_t stream);

/* ---- Cache append: the new token's rows written into the paged caches ------------ */
/* A decode step stores each new token's K-index row and latent row before the indexer
 * and the attention read them (both operators read the paged caches directly: "Day0
 * Inference Optimization on Ascend CANN", section 2).  Token i's rows go to page
 * block_table[b * max_pages_per_seq + pos / 64], slot pos % 64, with b = token_seq[i] (or
 * i) and pos = token_pos[i] (or seq_lens[b] - 1: the newest stored position).  A position
 * outside the page table sets DSA_DEVERR_TOKEN, a page id outside [0, num_pages)
 * DSA_DEVERR_PAGE_ID, in ws's error word; that token is skipped and the others are
 * written.  ws: 256-byte aligned, at least 256 bytes (only the error word is used; it
 * is not cleared by the call).  The cache structs' buffers are written, not only read.
 *
 * FP8 formats use absmax block quantisation (the pages leave the rule open): a block's
 * f32 scale is amax / 448 (amax: its largest magnitude; 448: the largest E4M3 value),
 * computed as an IEEE binary32 division, or 1 for an all-zero block; each element is
 * stored as the E4M3 value nearest to the binary32 quotient x / scale, ties to even,
 * saturating at +-448.  Inputs must be finite. */

/* K-index rows: device k_new bf16 [T, cache->dim] (16-byte aligned) into `cache`: bf16
 * (copied), e4m3 with DSA_SCALE_PER_TOKEN_F32 (one block per row: codes to data, the
 * scale to scale[page, slot]) or e4m3 with DSA_SCALE_MX_E8M0_G32 (as
 * dsa_index_cache_append_mxfp8). */
dsa_status_t dsa_index_cache_append(const void* k_new, const dsa_index_cache_t* cache,
                                    const dsa_page_table_t* pages, const dsa_tokens_t* tokens,
                                    void* ws, size_t ws_bytes, dsa_stream_t stream);

/* Latent rows: device rows_new bf16 [T, cache->dim] (16-byte aligned) into `cache`: bf16
 * (copied) or FP8 (each 128-dim latent tile a block: codes to data, scales to scale; the
 * rope dims copied to rope). */
dsa_status_t dsa_latent_cache_append(const void* rows_new, const dsa_latent_cache_t* cache,
                                     const dsa_page_table_t* pages, const dsa_tokens_t* tokens,
                                     void* ws, size_t ws_bytes, dsa_stream_t stream);

/* ---- Test hook: the indexer's pipeline wait limit ------------------------------- */
/* Every wait inside the indexer's tensor-core kernels (a TMA load landing, an MMA
 * completing, an epilogue freeing an accumulator) gives up after a limit -- about 2 s of
 * SM clock cycles by default -- and then sets DSA_DEVERR_TIMEOUT in the workspace's error
 * word, lets its in-flight copies and MMAs finish, frees its tensor memory and returns,
 * so a lost arrival never hangs the device.  This sets that limit, process-wide, for the
 * indexer calls launched afterwards (cycles > 0), or restores the default (0); a test
 * lowers it to a few hundred cycles to make ordinary waits run out.  The attention
 * kernel keeps its fixed limit (its CTA pairs exchange data through distributed shared
 * memory, and a CTA must not exit while its peer's copies into it are in flight).
 * Returns DSA_ERR_INVALID_ARG for cycles < 0. */
dsa_status_t dsa_set_indexer_wait_limit(int64_t cycles);

/* ---- Errors and introspection --------------------------------------------------- */
/* Copies the device error word out of ws (synchronises `stream`) into *err. */
dsa_status_t dsa_read_device_error(const void* ws, uint32_t* err, dsa_stream_t stream);
/* Zeroes the device error word (enqueued on `stream`). */
dsa_status_t dsa_clear_device_error(void* ws, dsa_stream_t stream);
const char* dsa_status_string(dsa_status_t s);
const char* dsa_last_error_message(void);
int32_t dsa_abi_version(void);

#ifdef __cplusplus
}
#endif
#endif /* DSA_GB300_DSA_H */
