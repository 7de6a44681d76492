// Host side of the C ABI declared in include/dsa.h: argument checks, launch planning,
// workspace carving and kernel launches.  No allocation, no host synchronisation
// except in dsa_read_device_error().
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <atomic>
#include <string>

#include "common.cuh"
#include "dsa_internal.h"

namespace dsa {
namespace {

thread_local std::string g_last_error;

// Pipeline wait limit of the indexer's tensor-core kernels (cycles; 0: the default, about
// 2 s).  Lowered only by tests, through dsa_set_indexer_wait_limit.
std::atomic<long long> g_indexer_wait_limit{0};

dsa_status_t fail(dsa_status_t st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return st;
}

dsa_status_t cuda_fail(cudaError_t e, const char* what) {
  return fail(DSA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

constexpr size_t kAlign = 256;
size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }
bool aligned16(const void* ptr) { return ((uintptr_t)ptr & 15u) == 0; }


// ---- shared checks -------------------------------------------------------------------
dsa_status_t check_pages_tokens(const dsa_page_table_t* pg, const dsa_tokens_t* tk, int32_t* max_visible) {
  if (!pg || !tk) return fail(DSA_ERR_INVALID_ARG, "page table or tokens is NULL");
  if (pg->page_size != kPage) return fail(DSA_ERR_UNSUPPORTED, "page_size must be 64 (got %d)", pg->page_size);
  if (pg->batch < 1 || pg->max_pages_per_seq < 1 || pg->num_pages < 1)
    return fail(DSA_ERR_INVALID_ARG, "batch, max_pages_per_seq and num_pages must be >= 1");
  if (!pg->block_table || !pg->seq_lens || !pg->seq_lens_host)
    return fail(DSA_ERR_INVALID_ARG, "block_table, seq_lens and seq_lens_host are required");
  if (tk->n_tokens < 1) return fail(DSA_ERR_INVALID_ARG, "n_tokens must be >= 1");
  if (!tk->token_seq && tk->n_tokens != pg->batch)
    return fail(DSA_ERR_INVALID_ARG, "token_seq NULL requires n_tokens == batch");
  if (tk->token_seq && !tk->token_seq_host)
    return fail(DSA_ERR_INVALID_ARG, "token_seq_host is required with token_seq");
  if (tk->token_pos && !tk->token_pos_host)
    return fail(DSA_ERR_INVALID_ARG, "token_pos_host is required with token_pos");
  const int64_t cap = (int64_t)pg->max_pages_per_seq * kPage;
  for (int b = 0; b < pg->batch; ++b) {
    const int32_t L = pg->seq_lens_host[b];
    if (L < 0 || L > cap)
      return fail(DSA_ERR_INVALID_ARG, "seq_lens_host[%d] = %d outside [0, %lld]", b, L, (long long)cap);
  }
  int32_t mv = 0;
  for (int i = 0; i < tk->n_tokens; ++i) {
    const int b = tk->token_seq ? tk->token_seq_host[i] : i;
    if (b < 0 || b >= pg->batch) return fail(DSA_ERR_INVALID_ARG, "token_seq_host[%d] = %d outside [0, batch)", i, b);
    const int32_t L = pg->seq_lens_host[b];
    const int32_t pos = tk->token_pos ? tk->token_pos_host[i] : L - 1;
    if (pos < -1) return fail(DSA_ERR_INVALID_ARG, "token_pos_host[%d] = %d < -1", i, pos);
    const int32_t n = pos + 1 < L ? pos + 1 : L;
    if (n > mv) mv = n;
  }
  if (mv > kMaxVisible)
    return fail(DSA_ERR_UNSUPPORTED, "a token sees %d positions; this build selects from at most %d", mv, kMaxVisible);
  *max_visible = mv;
  return DSA_OK;
}

TokenView token_view(const dsa_page_table_t* pg, const dsa_tokens_t* tk, int32_t max_visible) {
  TokenView tv;
  tv.max_visible = max_visible;
  tv.token_seq = tk->token_seq;
  tv.token_pos = tk->token_pos;
  tv.seq_lens = pg->seq_lens;
  tv.block_table = pg->block_table;
  tv.batch = pg->batch;
  tv.max_pages = pg->max_pages_per_seq;
  tv.num_pages = pg->num_pages;
  tv.n_tokens = tk->n_tokens;
  return tv;
}

dsa_status_t check_indexer(const dsa_indexer_args_t* a, const dsa_index_cache_t* c) {
  if (!a || !c) return fail(DSA_ERR_INVALID_ARG, "indexer args or cache is NULL");
  if (!a->q || !a->head_w || !c->data) return fail(DSA_ERR_INVALID_ARG, "q, head_w and cache data are required");
  if (a->n_heads < 1 || a->n_heads > kMaxIdxHeads)
    return fail(DSA_ERR_UNSUPPORTED, "indexer n_heads must be in [1, %d] (got %d)", kMaxIdxHeads, a->n_heads);
  if (c->dim != 64 && c->dim != 128) return fail(DSA_ERR_UNSUPPORTED, "index dim must be 64 or 128 (got %d)", c->dim);
  if (a->top_k < 1 || a->top_k > kMaxTopK)
    return fail(DSA_ERR_UNSUPPORTED, "top_k must be in [1, %d] (got %d)", kMaxTopK, a->top_k);
  if (a->act != DSA_ACT_IDENTITY && a->act != DSA_ACT_RELU) return fail(DSA_ERR_INVALID_ARG, "unknown activation");
  if (a->q_dtype != c->dtype || a->q_scale_kind != c->scale_kind)
    return fail(DSA_ERR_UNSUPPORTED, "query and cache must share dtype and scale kind");
  if (!aligned16(c->data) || (c->scale && !aligned16(c->scale)))
    return fail(DSA_ERR_INVALID_ARG, "index cache data and scales must be 16-byte aligned");
  if (c->dtype == DSA_BF16) {
    if (c->scale_kind != DSA_SCALE_NONE) return fail(DSA_ERR_UNSUPPORTED, "bf16 index cache takes no scales");
  } else if (c->dtype == DSA_E4M3) {
    if (c->scale_kind != DSA_SCALE_PER_TOKEN_F32 && c->scale_kind != DSA_SCALE_MX_E8M0_G32)
      return fail(DSA_ERR_UNSUPPORTED, "e4m3 index cache needs per-token f32 or MX E8M0 scales");
    if (!c->scale || !a->q_scale) return fail(DSA_ERR_INVALID_ARG, "e4m3 modes need q_scale and cache scale");
  } else {
    return fail(DSA_ERR_INVALID_ARG, "unknown index dtype");
  }
  return DSA_OK;
}

dsa_status_t check_sfa(const dsa_sfa_args_t* a, const dsa_latent_cache_t* c) {
  if (!a) return fail(DSA_ERR_INVALID_ARG, "sfa args is NULL");
  if (!a->q) return fail(DSA_ERR_INVALID_ARG, "sfa q is NULL");
  if (a->n_heads < 1 || a->n_heads > kMaxSfaHeads)
    return fail(DSA_ERR_UNSUPPORTED, "sfa n_heads must be in [1, %d] (got %d)", kMaxSfaHeads, a->n_heads);
  if (!std::isfinite(a->softmax_scale)) return fail(DSA_ERR_INVALID_ARG, "softmax_scale must be finite");
  if (!aligned16(a->q)) return fail(DSA_ERR_INVALID_ARG, "sfa q must be 16-byte aligned");
  if (c) {
    if (!c->data) return fail(DSA_ERR_INVALID_ARG, "latent cache data is NULL");
    if (!aligned16(c->data)) return fail(DSA_ERR_INVALID_ARG, "latent cache data must be 16-byte aligned");
    if (c->dim != kLatentDim || c->v_dim != kValueDim)
      return fail(DSA_ERR_UNSUPPORTED, "latent rows must be 576 wide with a 512-wide value (got %d/%d)", c->dim, c->v_dim);
    if (c->dtype == DSA_E4M3) {
      if (!c->scale || !c->rope) return fail(DSA_ERR_INVALID_ARG, "an FP8 latent cache needs scale and rope");
      if (!aligned16(c->scale) || !aligned16(c->rope))
        return fail(DSA_ERR_INVALID_ARG, "latent scales and rope must be 16-byte aligned");
    } else if (c->dtype != DSA_BF16) {
      return fail(DSA_ERR_INVALID_ARG, "unknown latent dtype");
    }
  }
  return DSA_OK;
}

// ---- zeroing (histograms, split counters) --------------------------------------------
// A kernel rather than a memset so that it takes part in programmatic dependent launch:
// it waits for the previous kernel (which may still use this workspace) and lets the
// next one start its set-up meanwhile.
__global__ void __launch_bounds__(256) clear_kernel(uint4* p, size_t n16) {
  pdl_trigger();
  pdl_wait();
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n16; i += (size_t)gridDim.x * blockDim.x)
    p[i] = make_uint4(0u, 0u, 0u, 0u);
}

// ---- workspace plans ------------------------------------------------------------------
// Workspace: [0, 256) the device error word; then one region the passes use in turn (the
// indexer's key histograms and score rows, later the attention's split partials).
// Which scoring kernel serves the call.  Row-blocked: identity activation and tokens in
// segments of consecutive rows of one sequence (a prefill: one segment; multi-token
// decode: each sequence's draft tokens, all segments of one length), so that the rows of
// a segment share each key tile; e4m3 keys take it only for a single sequence with many
// rows (a prefill), after an exact dequantisation of its pages to bf16.  Otherwise one
// row per query token.
enum class Route { kPerRow, kBlocked, kBlockedDequant };
struct IndexerRoute {
  Route route = Route::kPerRow;
  int32_t seg_rows = 1;  // row-blocked: rows per segment
  int32_t seq = 0;       // dequantised: the one sequence
};

IndexerRoute route_indexer(const dsa_indexer_args_t* a, const dsa_index_cache_t* c, const dsa_tokens_t* tk) {
  IndexerRoute rt;
  const int T = tk->n_tokens;
  if (a->act != DSA_ACT_IDENTITY || T < 2) return rt;
  auto seq = [&](int i) { return tk->token_seq ? tk->token_seq_host[i] : i; };
  int m = 1;
  while (m < T && seq(m) == seq(0)) ++m;
  const bool one_seq = m == T;
  bool uniform = m >= 2 && T % m == 0 && (one_seq || m <= kBlockedMaxSeg);
  for (int i = m; uniform && i < T; ++i)  // every later run of m rows is one sequence
    uniform = i % m == 0 || seq(i) == seq(i - 1);
  if (!uniform) return rt;
  if (c->dtype == DSA_BF16) {
    rt.route = Route::kBlocked;
  } else if (one_seq && T >= 2 * kBlockRows) {
    rt.route = Route::kBlockedDequant;
    rt.seq = seq(0);
  } else {
    return rt;
  }
  rt.seg_rows = m;
  return rt;
}

struct IndexerPlan {
  int32_t max_visible;
  int64_t score_stride;
  size_t score_bytes;  // the per-row key histograms, the collapsed query, the f32 score rows
                       // and, when dequantising, the bf16 keys, their scales and page table
  size_t hist_bytes, qt_bytes, rows_bytes;
  size_t kb_bytes = 0, ks_bytes = 0, bt_bytes = 0;  // dequantised keys (row-blocked e4m3)
  int32_t npv = 0;                                  // pages dequantised
  IndexerRoute rt;
};

IndexerPlan plan_indexer(int32_t max_visible, int32_t n_tokens, int32_t dim, const IndexerRoute& rt = IndexerRoute(),
                         const dsa_page_table_t* pg = nullptr) {
  IndexerPlan p;
  p.rt = rt;
  p.max_visible = max_visible;
  p.score_stride = ((int64_t)max_visible + 63) / 64 * 64;
  if (p.score_stride == 0) p.score_stride = 64;
  const size_t rows = align_up((size_t)n_tokens * p.score_stride * sizeof(float));
  p.hist_bytes = align_up((size_t)n_tokens * kTopkBins * sizeof(uint32_t));
  // collapsed-query scratch: f32 [T, dim] (folded query) or bf16 [T, 3, dim] (its split for
  // the row-blocked tensor-core path), sized as bf16 [T, 16, dim] + f32 [T, 16] (the
  // workspace formula the boundary documents)
  p.qt_bytes = align_up((size_t)n_tokens * kSplitQueryHeads * dim * sizeof(uint16_t)) +
               align_up((size_t)n_tokens * kSplitQueryHeads * sizeof(float));
  p.rows_bytes = rows;
  p.score_bytes = p.hist_bytes + p.qt_bytes + rows;
  if (rt.route == Route::kBlockedDequant && pg) {
    p.npv = (max_visible + kPage - 1) / kPage;
    p.kb_bytes = align_up((size_t)p.npv * kPage * dim * sizeof(uint16_t));
    p.ks_bytes = align_up((size_t)p.npv * kPage * sizeof(float));
    p.bt_bytes = align_up((size_t)pg->batch * pg->max_pages_per_seq * sizeof(int32_t));
    p.score_bytes += p.kb_bytes + p.ks_bytes + p.bt_bytes;
  }
  return p;
}

IndexerPlan plan_indexer(const dsa_indexer_args_t* a, const dsa_index_cache_t* c, const dsa_page_table_t* pg,
                         const dsa_tokens_t* tk, int32_t max_visible) {
  return plan_indexer(max_visible, tk->n_tokens, c->dim, route_indexer(a, c, tk), pg);
}

struct SfaPlan {
  int32_t n_splits, split_len;
  bool sib_merge;                      // two splits merged inside their cluster
  size_t part_o_bytes, part_lse_bytes;  // in the shared region (more than two splits)
  size_t region_bytes() const { return part_o_bytes + part_lse_bytes; }
};

SfaPlan plan_sfa(int32_t n_tokens, int32_t n_heads, int32_t top_k) {
  SfaPlan p;
  const int tiles = (top_k + 63) / 64;
  const int units = n_tokens * 2;  // one CTA pair per (token, split)
  int s = device_sm_count() / (units > 0 ? units : 1);
  if (s < 1) s = 1;
  if (s > tiles) s = tiles;
  if (s > 16) s = 16;
  p.n_splits = s;
  p.split_len = (tiles + s - 1) / s * 64;
  p.n_splits = (tiles * 64 + p.split_len - 1) / p.split_len;  // drop empty splits
  p.sib_merge = p.n_splits == 2;
  if (p.n_splits > 1 && !p.sib_merge) {
    const size_t hp = (size_t)(n_heads + 3) / 4 * 4;  // head stride rounded up for 16-byte loads
    p.part_o_bytes = align_up((size_t)n_tokens * p.n_splits * hp * kValueDim * sizeof(float));
    p.part_lse_bytes = align_up((size_t)n_tokens * p.n_splits * 2 * hp * sizeof(float));
  } else {
    p.part_o_bytes = p.part_lse_bytes = 0;
  }
  return p;
}

dsa_status_t check_ws(void* ws, size_t ws_bytes, size_t need) {
  if (!ws) return fail(DSA_ERR_WORKSPACE, "workspace is NULL");
  if (((uintptr_t)ws) % kAlign) return fail(DSA_ERR_WORKSPACE, "workspace must be 256-byte aligned");
  if (ws_bytes < need)
    return fail(DSA_ERR_WORKSPACE, "workspace of %zu bytes is below the %zu needed", ws_bytes, need);
  return DSA_OK;
}

// ---- tracing -----------------------------------------------------------------------
struct Tracer {
  dsa_trace_t* t;
  cudaStream_t s;
  int n = 0;
  explicit Tracer(dsa_trace_t* tr, cudaStream_t st) : t(tr), s(st) {
    if (t) t->n_recorded = 0;
  }
  cudaError_t status = cudaSuccess;
  void begin() {
    if (t && n < DSA_TRACE_MAX && t->begin[n]) note(cudaEventRecord((cudaEvent_t)t->begin[n], s));
  }
  void end(const char* name) {
    if (t && n < DSA_TRACE_MAX) {
      if (t->end[n]) note(cudaEventRecord((cudaEvent_t)t->end[n], s));
      t->name[n] = name;
      t->n_recorded = ++n;
    }
  }
  void note(cudaError_t e) {
    if (status == cudaSuccess) status = e;
  }
};

// ---- the three passes -----------------------------------------------------------------
// `region`: the pass region (histograms first); `clear` / `clear_bytes`: what to zero
// before the score kernel (the histograms, plus the split counters that precede them
// when the attention pass follows).
dsa_status_t run_indexer(const dsa_indexer_args_t* a, const dsa_index_cache_t* c,
                         const dsa_page_table_t* pg, const dsa_tokens_t* tk, const IndexerPlan& ip,
                         int32_t* out_idx, float* out_score, uint32_t* err, uint8_t* region, void* clear,
                         size_t clear_bytes, cudaStream_t s, Tracer& tr) {
  uint32_t* hist = (uint32_t*)region;
  float* qt = (float*)(region + ip.hist_bytes);
  uint16_t* qsplit = (uint16_t*)(region + ip.hist_bytes);  // (same scratch: the blocked path's split query)
  float* scores = (float*)(region + ip.hist_bytes + ip.qt_bytes);
  uint8_t* dq = region + ip.hist_bytes + ip.qt_bytes + ip.rows_bytes;  // dequantised keys (if any)
  ScoreParams sp;
  sp.tv = token_view(pg, tk, ip.max_visible);
  sp.q = a->q;
  sp.q_scale = a->q_scale;
  sp.head_w = a->head_w;
  sp.k = c->data;
  sp.k_scale = c->scale;
  sp.scores = scores;
  sp.hist = hist;
  sp.score_stride = ip.score_stride;
  sp.err = err;
  sp.n_heads = a->n_heads;
  sp.dim = c->dim;
  sp.act = (int)a->act;
  sp.max_page_blocks = (ip.max_visible + kPage - 1) / kPage;
  sp.q_dep = 0;
  {
    const long long wl = g_indexer_wait_limit.load(std::memory_order_relaxed);
    sp.wait_limit = wl > 0 ? wl : sm100_default_wait_limit();
  }
  tr.begin();
  cudaError_t me = launch_clear(clear, clear_bytes, s);
  tr.end("hist_clear");
  if (me != cudaSuccess) return cuda_fail(me, "clearing the key histograms");
  if (sp.max_page_blocks > 0) {
    // Otherwise the per-head contraction on the tensor cores (CUDA cores for shapes they
    // do not take).
    const bool identity = a->act == DSA_ACT_IDENTITY;
    // Query rows that share one sequence (a prefill, or a sequence's draft tokens) share
    // their keys: blocks of those rows take each K tile together (route_indexer).
    const bool blocked = ip.rt.route != Route::kPerRow;
    // e4m3 keys (per-token scales, d = 128) with the identity activation: the head
    // sum folds into the query, and each key is one dot product taken from the TMA-staged
    // tile on the CUDA cores.
    const bool fold = score_fold_supported(c->dtype, c->scale_kind, a->act, c->dim);
    const bool stream = !fold && identity && c->dtype == DSA_E4M3 &&
                        c->scale_kind == DSA_SCALE_PER_TOKEN_F32 && score_stream_supported(a->act, c->dim);
    const bool tc = score_tc_supported(c->dtype, c->dim, a->n_heads);
    tr.begin();
    cudaError_t e = cudaSuccess;
    if (blocked) {
      ScoreParams sp2 = sp;
      sp2.seg_rows = ip.rt.seg_rows;
      if (ip.rt.route == Route::kBlockedDequant) {
        uint16_t* kb = (uint16_t*)dq;
        float* ks = (float*)(dq + ip.kb_bytes);
        int32_t* bt = (int32_t*)(dq + ip.kb_bytes + ip.ks_bytes);
        e = launch_kdequant(sp, c->scale_kind, ip.rt.seq, ip.npv, kb, ks, bt, s);
        sp2.k = kb;
        sp2.k_scale = c->scale_kind == DSA_SCALE_PER_TOKEN_F32 ? ks : nullptr;
        sp2.tv.block_table = bt;
        sp2.tv.num_pages = ip.npv;
      }
      if (e == cudaSuccess) e = launch_qsplit(sp, c->dtype, c->scale_kind, qsplit, nullptr, 3, s);
      sp2.q = qsplit;
      sp2.q_dep = 1;
      if (e == cudaSuccess) e = launch_score_tc_blocked(sp2, s);
    } else if (fold) {
      e = launch_qtilde(sp, c->dtype, c->scale_kind, qt, s);
      if (e == cudaSuccess) e = launch_score_fold(sp, c->scale_kind, qt, s);
    } else {
      e = stream ? launch_score_stream(sp, c->dtype, c->scale_kind, qt, s)
          : tc   ? launch_score_tc(sp, c->dtype, c->scale_kind, s)
                 : launch_score(sp, c->dtype, c->scale_kind, s);
    }
    tr.end("indexer_score");
    if (e != cudaSuccess) return cuda_fail(e, "indexer score launch");
  }
  TopkParams tp;
  tp.tv = sp.tv;
  tp.scores = scores;
  tp.hist = hist;
  tp.score_stride = ip.score_stride;
  tp.out_idx = out_idx;
  tp.out_score = out_score;
  tp.err = err;
  tp.top_k = a->top_k;
  tr.begin();
  cudaError_t e = launch_topk(tp, ip.max_visible, s);
  tr.end("indexer_topk");
  if (e != cudaSuccess) return cuda_fail(e, "top-k launch");
  return DSA_OK;
}

// `region`: the pass region for the split partials.
dsa_status_t run_sfa(const dsa_sfa_args_t* a, const dsa_latent_cache_t* c, const dsa_page_table_t* pg,
                     const dsa_tokens_t* tk, int32_t max_visible, const int32_t* idx, int32_t top_k, void* out,
                     uint32_t* err, uint8_t* region, const SfaPlan& sp_, cudaStream_t s, Tracer& tr) {
  SfaParams p;
  p.tv = token_view(pg, tk, max_visible);
  p.q = (const uint16_t*)a->q;
  const bool fp8 = c->dtype == DSA_E4M3;
  p.kv = fp8 ? nullptr : (const uint16_t*)c->data;
  p.kv_codes = fp8 ? (const uint8_t*)c->data : nullptr;
  p.kv_scale = fp8 ? (const float*)c->scale : nullptr;
  p.kv_rope = fp8 ? (const uint16_t*)c->rope : nullptr;
  p.idx = idx;
  p.out = (uint16_t*)out;
  const bool global_merge = sp_.n_splits > 1 && !sp_.sib_merge;
  p.part_o = global_merge ? (float*)region : nullptr;
  p.part_lse = global_merge ? (float*)(region + sp_.part_o_bytes) : nullptr;
  p.sib_merge = sp_.sib_merge ? 1 : 0;
  p.err = err;
  p.n_heads = a->n_heads;
  p.top_k = top_k;
  p.n_splits = sp_.n_splits;
  p.split_len = sp_.split_len;
  p.scale_log2 = a->softmax_scale * 1.4426950408889634f;
  tr.begin();
  cudaError_t e = launch_sfa_tc(p, s);
  tr.end("sfa");
  if (e != cudaSuccess) return cuda_fail(e, "sparse attention launch");
  if (global_merge) {
    tr.begin();
    e = launch_sfa_combine(p, s);
    tr.end("sfa_combine");
    if (e != cudaSuccess) return cuda_fail(e, "split combine launch");
  }
  return DSA_OK;
}

}  // namespace

int device_sm_count() {
  // one lookup per device (an attribute query on every call would cost host time on the
  // launch path); entries are written once with the same value, so a race is harmless
  static std::atomic<int> cache[kMaxDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 148;
  int n = cache[dev].load(std::memory_order_relaxed);
  if (n > 0) return n;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 148;
  cache[dev].store(n, std::memory_order_relaxed);
  return n;
}

cudaError_t launch_clear(void* p, size_t bytes, cudaStream_t s) {
  const size_t n16 = bytes / 16;
  if (n16 == 0) return cudaSuccess;
  const unsigned blocks = (unsigned)(n16 < (size_t)256 * 4 * 152 ? (n16 + 1023) / 1024 : 4 * 152);
  return launch_pdl(clear_kernel, dim3(blocks), dim3(256), 0, s, (uint4*)p, n16);
}

}  // namespace dsa

using namespace dsa;

extern "C" {

size_t dsa_indexer_workspace_size(const dsa_indexer_args_t* args, const dsa_index_cache_t* cache,
                                  const dsa_page_table_t* pages, const dsa_tokens_t* tokens) {
  int32_t mv = 0;
  if (check_indexer(args, cache) != DSA_OK || check_pages_tokens(pages, tokens, &mv) != DSA_OK) return 0;
  return kAlign + plan_indexer(args, cache, pages, tokens, mv).score_bytes;
}

dsa_status_t dsa_indexer_topk(const dsa_indexer_args_t* args, const dsa_index_cache_t* cache,
                              const dsa_page_table_t* pages, const dsa_tokens_t* tokens, int32_t* out_idx,
                              float* out_score, void* ws, size_t ws_bytes, dsa_stream_t stream,
                              dsa_trace_t* trace) {
  dsa_status_t st = check_indexer(args, cache);
  if (st != DSA_OK) return st;
  int32_t mv = 0;
  if ((st = check_pages_tokens(pages, tokens, &mv)) != DSA_OK) return st;
  if (!out_idx) return fail(DSA_ERR_INVALID_ARG, "out_idx is NULL");
  IndexerPlan ip = plan_indexer(args, cache, pages, tokens, mv);
  if ((st = check_ws(ws, ws_bytes, kAlign + ip.score_bytes)) != DSA_OK) return st;
  Tracer tr(trace, (cudaStream_t)stream);
  uint8_t* region = (uint8_t*)ws + kAlign;
  st = run_indexer(args, cache, pages, tokens, ip, out_idx, out_score, (uint32_t*)ws, region, region, ip.hist_bytes,
                   (cudaStream_t)stream, tr);
  if (st == DSA_OK && tr.status != cudaSuccess) return cuda_fail(tr.status, "recording a trace event");
  return st;
}

size_t dsa_sparse_attn_workspace_size(const dsa_sfa_args_t* args, const dsa_page_table_t* pages,
                                      const dsa_tokens_t* tokens, int32_t top_k) {
  int32_t mv = 0;
  if (check_sfa(args, nullptr) != DSA_OK || check_pages_tokens(pages, tokens, &mv) != DSA_OK) return 0;
  if (top_k < 1 || top_k > kMaxTopK) return 0;
  SfaPlan sp = plan_sfa(tokens->n_tokens, args->n_heads, top_k);
  return kAlign + sp.region_bytes();
}

dsa_status_t dsa_sparse_attn(const dsa_sfa_args_t* args, const dsa_latent_cache_t* cache,
                             const dsa_page_table_t* pages, const dsa_tokens_t* tokens, const int32_t* idx,
                             int32_t top_k, void* out, void* ws, size_t ws_bytes, dsa_stream_t stream,
                             dsa_trace_t* trace) {
  dsa_status_t st = check_sfa(args, cache);
  if (st != DSA_OK) return st;
  if (!cache) return fail(DSA_ERR_INVALID_ARG, "latent cache is NULL");
  int32_t mv = 0;
  if ((st = check_pages_tokens(pages, tokens, &mv)) != DSA_OK) return st;
  if (!idx || !out) return fail(DSA_ERR_INVALID_ARG, "idx and out are required");
  if (!aligned16(out)) return fail(DSA_ERR_INVALID_ARG, "out must be 16-byte aligned");
  if (top_k < 1 || top_k > kMaxTopK) return fail(DSA_ERR_UNSUPPORTED, "top_k must be in [1, %d]", kMaxTopK);
  SfaPlan sp = plan_sfa(tokens->n_tokens, args->n_heads, top_k);
  if ((st = check_ws(ws, ws_bytes, kAlign + sp.region_bytes())) != DSA_OK) return st;
  Tracer tr(trace, (cudaStream_t)stream);
  uint8_t* w8 = (uint8_t*)ws;
  st = run_sfa(args, cache, pages, tokens, mv, idx, top_k, out, (uint32_t*)ws, w8 + kAlign, sp, (cudaStream_t)stream,
               tr);
  if (st == DSA_OK && tr.status != cudaSuccess) return cuda_fail(tr.status, "recording a trace event");
  return st;
}

size_t dsa_fused_workspace_size(const dsa_indexer_args_t* iargs, const dsa_index_cache_t* icache,
                                const dsa_sfa_args_t* sargs, const dsa_page_table_t* pages,
                                const dsa_tokens_t* tokens) {
  int32_t mv = 0;
  if (check_indexer(iargs, icache) != DSA_OK || check_sfa(sargs, nullptr) != DSA_OK ||
      check_pages_tokens(pages, tokens, &mv) != DSA_OK)
    return 0;
  IndexerPlan ip = plan_indexer(iargs, icache, pages, tokens, mv);
  SfaPlan sp = plan_sfa(tokens->n_tokens, sargs->n_heads, iargs->top_k);
  const size_t sfa_b = sp.region_bytes();
  return kAlign + (ip.score_bytes > sfa_b ? ip.score_bytes : sfa_b);  // the passes reuse one region
}

dsa_status_t dsa_fused_decode(const dsa_indexer_args_t* iargs, const dsa_index_cache_t* icache,
                              const dsa_sfa_args_t* sargs, const dsa_latent_cache_t* lcache,
                              const dsa_page_table_t* pages, const dsa_tokens_t* tokens, int32_t* out_idx,
                              void* out, void* ws, size_t ws_bytes, dsa_stream_t stream, dsa_trace_t* trace) {
  dsa_status_t st = check_indexer(iargs, icache);
  if (st != DSA_OK) return st;
  if ((st = check_sfa(sargs, lcache)) != DSA_OK) return st;
  if (!lcache) return fail(DSA_ERR_INVALID_ARG, "latent cache is NULL");
  int32_t mv = 0;
  if ((st = check_pages_tokens(pages, tokens, &mv)) != DSA_OK) return st;
  if (!out_idx || !out) return fail(DSA_ERR_INVALID_ARG, "out_idx and out are required");
  if (!aligned16(out)) return fail(DSA_ERR_INVALID_ARG, "out must be 16-byte aligned");
  IndexerPlan ip = plan_indexer(iargs, icache, pages, tokens, mv);
  SfaPlan sp = plan_sfa(tokens->n_tokens, sargs->n_heads, iargs->top_k);
  const size_t sfa_b = sp.region_bytes();
  if ((st = check_ws(ws, ws_bytes, kAlign + (ip.score_bytes > sfa_b ? ip.score_bytes : sfa_b))) !=
      DSA_OK)
    return st;
  Tracer tr(trace, (cudaStream_t)stream);
  uint8_t* w8 = (uint8_t*)ws;
  uint8_t* region = w8 + kAlign;
  // the indexer's clear zeroes the key histograms at the start of the region
  if ((st = run_indexer(iargs, icache, pages, tokens, ip, out_idx, nullptr, (uint32_t*)ws, region, region,
                        ip.hist_bytes, (cudaStream_t)stream, tr)) != DSA_OK)
    return st;
  st = run_sfa(sargs, lcache, pages, tokens, mv, out_idx, iargs->top_k, out, (uint32_t*)ws, region, sp,
               (cudaStream_t)stream, tr);
  if (st == DSA_OK && tr.status != cudaSuccess) return cuda_fail(tr.status, "recording a trace event");
  return st;
}

dsa_status_t dsa_quantize_mxfp8(const void* x, int64_t n_rows, int32_t dim, void* codes, void* scales,
                                dsa_stream_t stream) {
  if (!x || !codes || !scales) return fail(DSA_ERR_INVALID_ARG, "x, codes and scales are required");
  if (n_rows < 0 || n_rows > INT32_MAX) return fail(DSA_ERR_INVALID_ARG, "n_rows = %lld outside [0, 2^31)", (long long)n_rows);
  if (dim < 32 || dim > 8192 || dim % 32)
    return fail(DSA_ERR_INVALID_ARG, "dim = %d: a multiple of 32 in [32, 8192]", dim);
  if (((uintptr_t)x) % 16 || ((uintptr_t)codes) % 8)
    return fail(DSA_ERR_INVALID_ARG, "x must be 16-byte and codes 8-byte aligned");
  Mxfp8Params p{};
  p.x = (const uint16_t*)x;
  p.n_rows = n_rows;
  p.dim = dim;
  p.codes = (uint8_t*)codes;
  p.scales = (uint8_t*)scales;
  p.append = false;
  cudaError_t e = launch_mxfp8_quant(p, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "MXFP8 quantisation launch");
  return DSA_OK;
}

dsa_status_t dsa_index_cache_append_mxfp8(const void* k_new, int32_t dim, const dsa_page_table_t* pages,
                                          const dsa_tokens_t* tokens, void* cache_codes, void* cache_scales,
                                          void* ws, size_t ws_bytes, dsa_stream_t stream) {
  if (!k_new || !cache_codes || !cache_scales)
    return fail(DSA_ERR_INVALID_ARG, "k_new, cache_codes and cache_scales are required");
  if (dim != 64 && dim != 128) return fail(DSA_ERR_UNSUPPORTED, "dim must be 64 or 128 (got %d)", dim);
  if (((uintptr_t)k_new) % 16 || ((uintptr_t)cache_codes) % 16)
    return fail(DSA_ERR_INVALID_ARG, "k_new and cache_codes must be 16-byte aligned");
  int32_t mv = 0;
  dsa_status_t st = check_pages_tokens(pages, tokens, &mv);
  if (st != DSA_OK) return st;
  if ((st = check_ws(ws, ws_bytes, kAlign)) != DSA_OK) return st;
  Mxfp8Params p{};
  p.x = (const uint16_t*)k_new;
  p.n_rows = tokens->n_tokens;
  p.dim = dim;
  p.codes = (uint8_t*)cache_codes;
  p.scales = (uint8_t*)cache_scales;
  p.append = true;
  p.tv = token_view(pages, tokens, mv);
  p.err = (uint32_t*)ws;
  cudaError_t e = launch_mxfp8_quant(p, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "K-index append launch");
  return DSA_OK;
}

dsa_status_t dsa_index_cache_append(const void* k_new, const dsa_index_cache_t* cache, const dsa_page_table_t* pages,
                                    const dsa_tokens_t* tokens, void* ws, size_t ws_bytes, dsa_stream_t stream) {
  if (!cache) return fail(DSA_ERR_INVALID_ARG, "cache is NULL");
  if (cache->dtype == DSA_E4M3 && cache->scale_kind == DSA_SCALE_MX_E8M0_G32)
    return dsa_index_cache_append_mxfp8(k_new, cache->dim, pages, tokens, const_cast<void*>(cache->data),
                                        const_cast<void*>(cache->scale), ws, ws_bytes, stream);
  if (!k_new || !cache->data) return fail(DSA_ERR_INVALID_ARG, "k_new and cache data are required");
  if (cache->dim != 64 && cache->dim != 128) return fail(DSA_ERR_UNSUPPORTED, "dim must be 64 or 128 (got %d)", cache->dim);
  const bool fp8 = cache->dtype == DSA_E4M3;
  if (fp8 ? (cache->scale_kind != DSA_SCALE_PER_TOKEN_F32 || !cache->scale)
          : (cache->dtype != DSA_BF16 || cache->scale_kind != DSA_SCALE_NONE))
    return fail(DSA_ERR_UNSUPPORTED, "index cache format: bf16, or e4m3 with per-token f32 or MX scales");
  if (!aligned16(k_new) || !aligned16(cache->data) || (cache->scale && !aligned16(cache->scale)))
    return fail(DSA_ERR_INVALID_ARG, "k_new and the cache buffers must be 16-byte aligned");
  int32_t mv = 0;
  dsa_status_t st = check_pages_tokens(pages, tokens, &mv);
  if (st != DSA_OK) return st;
  if ((st = check_ws(ws, ws_bytes, kAlign)) != DSA_OK) return st;
  IndexAppendParams p{};
  p.x = (const uint16_t*)k_new;
  p.n_rows = tokens->n_tokens;
  p.data = const_cast<void*>(cache->data);
  p.scales = (float*)const_cast<void*>(cache->scale);
  p.tv = token_view(pages, tokens, mv);
  p.err = (uint32_t*)ws;
  cudaError_t e = launch_index_append(p, cache->dim, fp8, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "K-index append launch");
  return DSA_OK;
}

dsa_status_t dsa_latent_cache_append(const void* rows_new, const dsa_latent_cache_t* cache,
                                     const dsa_page_table_t* pages, const dsa_tokens_t* tokens, void* ws,
                                     size_t ws_bytes, dsa_stream_t stream) {
  if (!rows_new || !cache || !cache->data) return fail(DSA_ERR_INVALID_ARG, "rows_new and cache data are required");
  if (cache->dim != kLatentDim || cache->v_dim != kValueDim)
    return fail(DSA_ERR_UNSUPPORTED, "latent rows must be 576 wide with a 512-wide value (got %d/%d)", cache->dim,
                cache->v_dim);
  const bool fp8 = cache->dtype == DSA_E4M3;
  if (!fp8 && cache->dtype != DSA_BF16) return fail(DSA_ERR_INVALID_ARG, "unknown latent dtype");
  if (fp8 && (!cache->scale || !cache->rope)) return fail(DSA_ERR_INVALID_ARG, "an FP8 latent cache needs scale and rope");
  if (!aligned16(rows_new) || !aligned16(cache->data) || (fp8 && (!aligned16(cache->scale) || !aligned16(cache->rope))))
    return fail(DSA_ERR_INVALID_ARG, "rows_new and the cache buffers must be 16-byte aligned");
  int32_t mv = 0;
  dsa_status_t st = check_pages_tokens(pages, tokens, &mv);
  if (st != DSA_OK) return st;
  if ((st = check_ws(ws, ws_bytes, kAlign)) != DSA_OK) return st;
  LatentAppendParams p{};
  p.x = (const uint16_t*)rows_new;
  p.n_rows = tokens->n_tokens;
  p.data = fp8 ? nullptr : (uint16_t*)const_cast<void*>(cache->data);
  p.codes = fp8 ? (uint8_t*)const_cast<void*>(cache->data) : nullptr;
  p.scales = fp8 ? (float*)const_cast<void*>(cache->scale) : nullptr;
  p.rope = fp8 ? (uint16_t*)const_cast<void*>(cache->rope) : nullptr;
  p.tv = token_view(pages, tokens, mv);
  p.err = (uint32_t*)ws;
  cudaError_t e = launch_latent_append(p, fp8, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "latent append launch");
  return DSA_OK;
}

dsa_status_t dsa_set_indexer_wait_limit(int64_t cycles) {
  if (cycles < 0) return fail(DSA_ERR_INVALID_ARG, "cycles must be >= 0 (0 restores the default)");
  g_indexer_wait_limit.store(cycles, std::memory_order_relaxed);
  return DSA_OK;
}

dsa_status_t dsa_read_device_error(const void* ws, uint32_t* err, dsa_stream_t stream) {
  if (!ws || !err) return fail(DSA_ERR_INVALID_ARG, "ws and err are required");
  cudaError_t e = cudaMemcpyAsync(err, ws, sizeof(uint32_t), cudaMemcpyDeviceToHost, (cudaStream_t)stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize((cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "reading the device error word");
  return DSA_OK;
}

dsa_status_t dsa_clear_device_error(void* ws, dsa_stream_t stream) {
  if (!ws) return fail(DSA_ERR_INVALID_ARG, "ws is NULL");
  cudaError_t e = cudaMemsetAsync(ws, 0, sizeof(uint32_t), (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "clearing the device error word");
  return DSA_OK;
}

const char* dsa_status_string(dsa_status_t s) {
  switch (s) {
    case DSA_OK: return "DSA_OK";
    case DSA_ERR_INVALID_ARG: return "DSA_ERR_INVALID_ARG";
    case DSA_ERR_UNSUPPORTED: return "DSA_ERR_UNSUPPORTED";
    case DSA_ERR_WORKSPACE: return "DSA_ERR_WORKSPACE";
    case DSA_ERR_CUDA: return "DSA_ERR_CUDA";
  }
  return "DSA_ERR_UNKNOWN";
}

const char* dsa_last_error_message(void) { return g_last_error.c_str(); }

int32_t dsa_abi_version(void) { return DSA_ABI_VERSION; }

}  // extern "C"

// ---- indexer with the library's own fixed scratch ------------------------------------
// For callers that cannot allocate device memory.  The scratch is a fixed device array
// defined in noalloc.cu (its own module, so that it becomes resident on a device only
// when this entry point first looks up its address there, under lazy module loading).
extern "C" dsa_status_t dsa_indexer_topk_noalloc(const dsa_indexer_args_t* args, const dsa_index_cache_t* cache,
                                                 const dsa_page_table_t* pages, const dsa_tokens_t* tokens,
                                                 int32_t* out_idx, float* out_score, dsa_stream_t stream) {
  dsa_status_t st = check_indexer(args, cache);
  if (st != DSA_OK) return st;
  int32_t mv = 0;
  if ((st = check_pages_tokens(pages, tokens, &mv)) != DSA_OK) return st;
  if (!out_idx) return fail(DSA_ERR_INVALID_ARG, "out_idx is NULL");
  IndexerPlan ip = plan_indexer(args, cache, pages, tokens, mv);
  const size_t need = kAlign + ip.score_bytes;
  if (need > kNoAllocScratchBytes)
    return fail(DSA_ERR_WORKSPACE,
                "dsa_indexer_topk_noalloc needs %zu bytes of scratch; its fixed scratch holds %zu "
                "(use dsa_indexer_topk with a caller workspace)",
                need, kNoAllocScratchBytes);
  void* ws = nullptr;
  int dev = -1;
  const cudaError_t e = noalloc_scratch(&ws, &dev);
  if (e != cudaSuccess) return cuda_fail(e, "looking up the fixed scratch's device address");
  if (!ws) return fail(DSA_ERR_UNSUPPORTED, "device ordinal %d beyond the %d the fixed scratch covers", dev, kMaxDevices);
  // The error word at the start of the scratch is only ever OR-ed into by the kernels and
  // never read back through this entry point, so it is not cleared per call; the key
  // histograms are zeroed inside run_indexer.
  Tracer tr(nullptr, (cudaStream_t)stream);
  uint8_t* region = (uint8_t*)ws + kAlign;
  return run_indexer(args, cache, pages, tokens, ip, out_idx, out_score, (uint32_t*)ws, region, region,
                     ip.hist_bytes, (cudaStream_t)stream, tr);
}
