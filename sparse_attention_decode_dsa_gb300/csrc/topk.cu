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
// memory, and every CTA derives the same digit.  The output is then a stable compaction
// in position order: keys > T, plus the first (K - #{key > T}) keys equal to T.
#include <cooperative_groups.h>

#include "common.cuh"

namespace cg = cooperative_groups;

namespace dsa {

namespace {

constexpr int kTopkThreads = 512;
constexpr int kWarps = kTopkThreads / 32;

// Exclusive prefix count of `flag` over the CTA in thread order, and the CTA total.
__device__ __forceinline__ int block_excl_count(bool flag, int* warp_buf, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  unsigned bal = __ballot_sync(0xffffffffu, flag);
  int in_warp = __popc(bal & ((1u << lane) - 1u));
  __syncthreads();  // warp_buf may still be read by the previous call
  if (lane == 0) warp_buf[warp] = __popc(bal);
  __syncthreads();
  int before = 0, tot = 0;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    int c = warp_buf[w];
    before += (w < warp) ? c : 0;
    tot += c;
  }
  *total = tot;
  return before + in_warp;
}

__global__ void __cluster_dims__(kTopkCluster, 1, 1) __launch_bounds__(kTopkThreads)
    topk_cluster_kernel(TopkParams p) {
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = (int)cluster.block_rank();
  const int row = blockIdx.y;
  const int tid = threadIdx.x;
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

  extern __shared__ uint32_t keys[];
  __shared__ uint32_t hist[2][256];
  __shared__ uint32_t ghist[256];
  __shared__ int warp_buf[kWarps];
  __shared__ int cnt[2];            // this CTA's #{key > T}, #{key == T}
  __shared__ uint32_t s_digit, s_above;
  __shared__ int s_taken_before, s_eq_before;

  const int chunk = (n + kTopkCluster - 1) / kTopkCluster;
  const int lo = rank * chunk;
  const int hi = min(n, lo + chunk);
  const int len = max(0, hi - lo);
  const float* srow = p.scores + (int64_t)row * p.score_stride + lo;
  for (int i = tid; i < len; i += kTopkThreads) keys[i] = score_key(srow[i]);

  uint32_t prefix = 0, mask = 0;
  uint32_t remaining = (uint32_t)K;  // how many still to pick among keys matching prefix
  const int lane = tid & 31;
#pragma unroll 1
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    uint32_t* h = hist[pass & 1];
    for (int i = tid; i < 256; i += kTopkThreads) h[i] = 0;
    __syncthreads();
    for (int base = 0; base < len; base += kTopkThreads) {
      const int i = base + tid;
      const bool in = i < len && ((keys[i] & mask) == prefix);
      const uint32_t dgt = in ? ((keys[i] >> shift) & 0xFFu) : 0u;
      const unsigned act = __ballot_sync(0xffffffffu, in);
      if (in) {
        const unsigned peers = __match_any_sync(act, dgt);
        if (lane == __ffs(peers) - 1) atomicAdd(&h[dgt], (uint32_t)__popc(peers));
      }
    }
    cluster.sync();
    for (int i = tid; i < 256; i += kTopkThreads) {
      uint32_t tot = 0;
#pragma unroll
      for (int r = 0; r < kTopkCluster; ++r) tot += cluster.map_shared_rank(h, r)[i];
      ghist[i] = tot;
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
        uint32_t v = __shfl_up_sync(0xffffffffu, incl, o);
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
  }
  const uint32_t T = prefix;  // the K-th largest key; take `remaining` of the keys == T

  int n_gt = 0, n_eq = 0;
  for (int i = tid; i < len; i += kTopkThreads) {
    n_gt += keys[i] > T;
    n_eq += keys[i] == T;
  }
  for (int o = 16; o; o >>= 1) {
    n_gt += __shfl_xor_sync(0xffffffffu, n_gt, o);
    n_eq += __shfl_xor_sync(0xffffffffu, n_eq, o);
  }
  if (tid == 0) cnt[0] = cnt[1] = 0;
  __syncthreads();
  if (lane == 0) {
    atomicAdd(&cnt[0], n_gt);
    atomicAdd(&cnt[1], n_eq);
  }
  cluster.sync();
  if (tid == 0) {
    int taken = 0, eq_before = 0;
    for (int r = 0; r < rank; ++r) {
      const int* c = cluster.map_shared_rank(cnt, r);
      const int gt_r = c[0], eq_r = c[1];
      const int take_eq = max(0, min((int)remaining - eq_before, eq_r));
      taken += gt_r + take_eq;
      eq_before += eq_r;
    }
    s_taken_before = taken;
    s_eq_before = eq_before;
  }
  cluster.sync();  // no CTA leaves while another may still read its shared memory

  int taken = s_taken_before, ties_seen = s_eq_before;
  for (int base = 0; base < len; base += kTopkThreads) {
    const int i = base + tid;
    const uint32_t key = i < len ? keys[i] : 0u;
    const bool gt = i < len && key > T;
    const bool eq = i < len && key == T;
    int eq_total;
    const int eq_rank = ties_seen + block_excl_count(eq, warp_buf, &eq_total);
    const bool take = gt || (eq && eq_rank < (int)remaining);
    int tk_total;
    const int pos = taken + block_excl_count(take, warp_buf, &tk_total);
    if (take && pos < K) {
      out[pos] = lo + i;
      if (outs) outs[pos] = key_score(key);
    }
    taken += tk_total;
    ties_seen += eq_total;
  }
}

}  // namespace

cudaError_t launch_topk(const TopkParams& p, int32_t max_visible, cudaStream_t s) {
  const int chunk = (max_visible + kTopkCluster - 1) / kTopkCluster;
  const size_t smem = (size_t)(chunk > 0 ? chunk : 1) * sizeof(uint32_t);
  cudaError_t e = cudaFuncSetAttribute(topk_cluster_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid(kTopkCluster, p.tv.n_tokens);
  topk_cluster_kernel<<<grid, kTopkThreads, smem, s>>>(p);
  return cudaGetLastError();
}

}  // namespace dsa
