// Lightning Indexer, selection pass: Top-K of one score row per query token.
//
// "Adapting and Optimizing Inference for a New Model Architecture on Ascend", section
// 3.1 (``topk_select``) and "Day0 Inference Optimization for New LLM Architectures on
// Heterogeneous Computing Platforms", section 2.1 (scoring and selection "on-chip"):
// the K largest scores of a row, ties to the lower position, returned as ascending
// positions padded with -1.
//
// One thread-block cluster of kTopkCluster CTAs per row.  Each CTA keeps a contiguous
// chunk of the row as order-preserving 32-bit keys in shared memory.  An exact MSB-first
// radix select (four 8-bit digits) finds the K-th largest key T: every CTA builds the
// histogram of its chunk, the cluster sums the histograms through distributed shared
// memory, and every CTA derives the same digit.  After two digits only the keys that
// still share the prefix are kept for the last two.  The output is then a stable
// compaction in position order (each thread owns a contiguous segment): keys > T, plus
// the first (K - #{key > T}) keys equal to T.
#include <cooperative_groups.h>

#include "common.cuh"

namespace cg = cooperative_groups;

namespace dsa {

namespace {

constexpr int kTopkThreads = 256;
constexpr int kWarps = kTopkThreads / 32;
constexpr int kCandCap = 8192;  // keys kept for the last two digits (else all keys are rescanned)

// Keys live at padded positions so that a thread walking its own contiguous segment
// hits a different bank from its neighbours.
__host__ __device__ __forceinline__ int kpos(int i) { return i + (i >> 5); }

// Exclusive prefix sum of v over the CTA in thread order, and the CTA total.
__device__ __forceinline__ int block_excl_sum(int v, int* buf, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int u = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += u;
  }
  if (lane == 31) buf[warp] = incl;
  __syncthreads();
  int before = 0, tot = 0;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    const int c = buf[w];
    before += (w < warp) ? c : 0;
    tot += c;
  }
  __syncthreads();  // buf is reused by the next call
  *total = tot;
  return before + incl - v;
}

// Adds the digit histogram of one key (warp-aggregated over equal digits).
__device__ __forceinline__ void hist_add(uint32_t* h, bool in, uint32_t dgt, int lane) {
  const unsigned act = __ballot_sync(0xffffffffu, in);
  if (in) {
    const unsigned peers = __match_any_sync(act, dgt);
    if (lane == __ffs(peers) - 1) atomicAdd(&h[dgt], (uint32_t)__popc(peers));
  }
}

__global__ void __cluster_dims__(kTopkCluster, 1, 1) __launch_bounds__(kTopkThreads)
    topk_cluster_kernel(TopkParams p) {
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = (int)cluster.block_rank();
  const int row = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31;
  const int K = p.top_k;

  int b, n;
  resolve_token(p.tv, row, &b, &n, nullptr);  // the score pass reports bad metadata
  int32_t* out = p.out_idx + (int64_t)row * K;
  float* outs = p.out_score ? p.out_score + (int64_t)row * K : nullptr;

  if (n <= K) {  // every visible position is selected (uniform over the cluster)
    for (int i = rank * kTopkThreads + tid; i < K; i += kTopkCluster * kTopkThreads) {
      out[i] = i < n ? i : -1;
      if (outs) outs[i] = i < n ? p.scores[(int64_t)row * p.score_stride + i] : __uint_as_float(0x7FC00000u);
    }
    return;
  }

  extern __shared__ uint32_t dyn[];
  __shared__ uint32_t hist[2][256];
  __shared__ uint32_t ghist[256];
  __shared__ int buf[kWarps];
  __shared__ int cnt[2];  // this CTA's #{key > T}, #{key == T}
  __shared__ uint32_t s_digit, s_above;
  __shared__ int s_ncand, s_taken_before, s_eq_before;

  const int chunk = (n + kTopkCluster - 1) / kTopkCluster;
  const int lo = rank * chunk;
  const int len = max(0, min(n, lo + chunk) - lo);
  uint32_t* keys = dyn;                              // [kpos(chunk)]
  uint32_t* cand = dyn + kpos(chunk) + 1;            // [min(chunk, kCandCap)]
  const int cand_cap = min(chunk, kCandCap);
  const float* srow = p.scores + (int64_t)row * p.score_stride + lo;
  for (int i = tid; i < len; i += kTopkThreads) keys[kpos(i)] = score_key(srow[i]);
  if (tid == 0) s_ncand = 0;

  uint32_t prefix = 0, mask = 0;
  uint32_t remaining = (uint32_t)K;  // how many still to pick among keys matching prefix
  bool use_cand = false;
  int ncand = 0;
#pragma unroll 1
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    uint32_t* h = hist[pass & 1];
    h[tid] = 0;  // kTopkThreads == 256 bins
    __syncthreads();
    if (use_cand) {
      for (int base = 0; base < ncand; base += kTopkThreads) {
        const int i = base + tid;
        const uint32_t k = i < ncand ? cand[i] : 0u;
        hist_add(h, i < ncand && (k & mask) == prefix, (k >> shift) & 0xFFu, lane);
      }
    } else {
      for (int base = 0; base < len; base += kTopkThreads) {
        const int i = base + tid;
        const uint32_t k = i < len ? keys[kpos(i)] : 0u;
        hist_add(h, i < len && (k & mask) == prefix, (k >> shift) & 0xFFu, lane);
      }
    }
    cluster.sync();
    {
      uint32_t tot = 0;
#pragma unroll
      for (int r = 0; r < kTopkCluster; ++r) tot += cluster.map_shared_rank(h, r)[tid];
      ghist[tid] = tot;
    }
    __syncthreads();
    if (tid < 32) {
      // lane l owns bins 255-8l .. 248-8l (high to low)
      uint32_t local = 0;
#pragma unroll
      for (int u = 0; u < 8; ++u) local += ghist[255 - 8 * lane - u];
      uint32_t incl = local;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      const uint32_t excl = incl - local;
      if (excl < remaining && remaining <= incl) {
        uint32_t cum = excl;
        for (int u = 0; u < 8; ++u) {
          const int bin = 255 - 8 * lane - u;
          if (cum + ghist[bin] >= remaining) {
            s_digit = (uint32_t)bin;
            s_above = cum;
            break;
          }
          cum += ghist[bin];
        }
      }
    }
    __syncthreads();
    prefix |= s_digit << shift;
    mask |= 0xFFu << shift;
    remaining -= s_above;
    if (pass == 1) {
      // keep the keys that still match the 16-bit prefix for the last two digits
      for (int base = 0; base < len; base += kTopkThreads) {
        const int i = base + tid;
        const uint32_t k = i < len ? keys[kpos(i)] : 0u;
        const bool in = i < len && (k & mask) == prefix;
        const unsigned bal = __ballot_sync(0xffffffffu, in);
        int slot = 0;
        if (lane == 0 && bal) slot = atomicAdd(&s_ncand, __popc(bal));
        slot = __shfl_sync(0xffffffffu, slot, 0) + __popc(bal & ((1u << lane) - 1u));
        if (in && slot < cand_cap) cand[slot] = k;
      }
      __syncthreads();
      ncand = s_ncand;
      use_cand = ncand <= cand_cap;
    }
  }
  const uint32_t T = prefix;  // the K-th largest key; take `remaining` of the keys == T

  // ---- stable compaction: every thread walks a contiguous segment of the chunk ------
  const int seg = (len + kTopkThreads - 1) / kTopkThreads;
  const int s0 = min(len, tid * seg), s1 = min(len, s0 + seg);
  int n_gt = 0, n_eq = 0;
  for (int i = s0; i < s1; ++i) {
    const uint32_t k = keys[kpos(i)];
    n_gt += k > T;
    n_eq += k == T;
  }
  int eq_total, gt_total;
  const int eq_base = block_excl_sum(n_eq, buf, &eq_total);
  block_excl_sum(n_gt, buf, &gt_total);
  if (tid == 0) {
    cnt[0] = gt_total;
    cnt[1] = eq_total;
  }
  cluster.sync();
  if (tid == 0) {
    int taken = 0, eq_before = 0;
    for (int r = 0; r < rank; ++r) {
      const int* c = cluster.map_shared_rank(cnt, r);
      const int gt_r = c[0], eq_r = c[1];
      taken += gt_r + max(0, min((int)remaining - eq_before, eq_r));
      eq_before += eq_r;
    }
    s_taken_before = taken;
    s_eq_before = eq_before;
  }
  cluster.sync();  // no CTA leaves while another may still read its shared memory
  const int tie0 = s_eq_before + eq_base;  // ties before this thread's segment, row-wide
  const int my_eq = max(0, min((int)remaining - tie0, n_eq));
  int tk_total;
  int pos = s_taken_before + block_excl_sum(n_gt + my_eq, buf, &tk_total);
  int ties = tie0;
  for (int i = s0; i < s1; ++i) {
    const uint32_t k = keys[kpos(i)];
    bool take = k > T;
    if (k == T) take = ties++ < (int)remaining;
    if (take && pos < K) {
      out[pos] = lo + i;
      if (outs) outs[pos] = key_score(k);
      ++pos;
    }
  }
}

}  // namespace

cudaError_t launch_topk(const TopkParams& p, int32_t max_visible, cudaStream_t s) {
  int chunk = (max_visible + kTopkCluster - 1) / kTopkCluster;
  if (chunk < 1) chunk = 1;
  const size_t smem = (size_t)(kpos(chunk) + 1 + (chunk < kCandCap ? chunk : kCandCap)) * sizeof(uint32_t);
  cudaError_t e = cudaFuncSetAttribute(topk_cluster_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid(kTopkCluster, p.tv.n_tokens);
  topk_cluster_kernel<<<grid, kTopkThreads, smem, s>>>(p);
  return cudaGetLastError();
}

}  // namespace dsa
