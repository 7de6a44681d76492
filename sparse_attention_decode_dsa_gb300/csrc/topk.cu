// Lightning Indexer, selection pass: Top-K of one score row per query token.
//
// "Adapting and Optimizing Inference for a New Model Architecture on Ascend", section
// 3.1 (``topk_select``) and "Day0 Inference Optimization for New LLM Architectures on
// Heterogeneous Computing Platforms", section 2.1 (scoring and selection "on-chip"):
// the K largest scores of a row, ties to the lower position, returned as ascending
// positions padded with -1.
//
// Scores are compared through an order-preserving 32-bit key (score_key).  The scoring
// pass already counted, per row, how many keys fall in each of the 4096 bins of their
// top 12 bits (kept in the workspace).  A cluster of C CTAs (1, 2, 4 or 8: the fewest
// that keep a CTA's share of the longest row within 4096 keys; 16 for rows beyond 32768)
// shares each row, CTA r owning the r-th C-th of its positions:
//   1. every CTA finds, from that histogram, the bin holding the K-th largest key (its
//      own keys are loading meanwhile);
//   2. each CTA counts its keys above that bin and gathers the keys in it (the
//      candidates; each warp into its own slice);
//   3. each CTA writes its count and its candidates into every CTA's pool (distributed
//      shared memory); after one cluster barrier every CTA finds the same exact K-th
//      largest key T among all candidates with an MSB-first radix select over the
//      remaining 20 bits (10 + 10), and from the pool alone how many keys > T and
//      == T each CTA holds, hence where its output starts;
//   4. each CTA writes, in position order, its keys > T and its share of the first
//      (K - #{> T}) keys == T (warps own contiguous ranges; block scans place them).
// Keys are read from the score row (in L2) in blocks of 4096 positions held in
// registers, all loads of a block in flight together.  If a CTA has more candidates
// than its pool slot (a row with very many equal top bits), steps 3-4 fall back to a
// radix select over each CTA's own keys whose histograms and counts the cluster sums
// through distributed shared memory, with the same result.
#include <cooperative_groups.h>

#include <atomic>

#include "common.cuh"
#include "dsa_internal.h"

namespace cg = cooperative_groups;

namespace dsa {

namespace {

constexpr int kThreads = 256;
constexpr int kWarpsPerCta = kThreads / 32;
constexpr int kChunks = 16;                      // 32-position chunks per warp per block
constexpr int kBlock = kThreads * kChunks;       // positions whose keys sit in registers
constexpr int kLocalCap = 2048;                  // candidates one CTA may gather
constexpr int kPoolTotal = 2048;                 // pooled candidates of a row (kSlot per CTA)

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
  for (int w = 0; w < kWarpsPerCta; ++w) {
    const int c = buf[w];
    before += (w < warp) ? c : 0;
    tot += c;
  }
  __syncthreads();  // buf is reused by the next call
  *total = tot;
  return before + incl - v;
}

// Finds, over a 256-bin histogram (high to low), the bin holding the `remaining`-th
// largest entry; warp 0 writes the bin and the count above it.
__device__ __forceinline__ void find_bin256(const uint32_t* hist, uint32_t remaining, uint32_t* s_digit,
                                            uint32_t* s_above) {
  const int lane = threadIdx.x & 31;
  uint32_t loc = 0;
#pragma unroll
  for (int u = 0; u < 8; ++u) loc += hist[255 - 8 * lane - u];
  uint32_t incl = loc;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  const uint32_t ex = incl - loc;
  if (ex < remaining && remaining <= incl) {
    uint32_t cum = ex;
    for (int u = 0; u < 8; ++u) {
      const int bin = 255 - 8 * lane - u;
      if (cum + hist[bin] >= remaining) {
        *s_digit = (uint32_t)bin;
        *s_above = cum;
        break;
      }
      cum += hist[bin];
    }
  }
}

// Same over a 1024-bin histogram, by the whole CTA: thread t owns bins 1023 - 4t ..
// 1020 - 4t (one 16-byte load); a block scan places them.  Every thread calls it; it
// ends with a barrier after which s_digit / s_above hold the result.
__device__ __forceinline__ void find_bin1024(const uint32_t* hist, uint32_t remaining, int* buf,
                                             uint32_t* s_digit, uint32_t* s_above) {
  static_assert(kThreads * 4 == 1024, "four bins per thread");
  const int tid = threadIdx.x;
  const uint4 q = *(const uint4*)(hist + 1020 - 4 * tid);
  const uint32_t h[4] = {q.w, q.z, q.y, q.x};  // bins 1023 - 4t - u, high to low
  const uint32_t loc = h[0] + h[1] + h[2] + h[3];
  int tot;
  const uint32_t ex = (uint32_t)block_excl_sum((int)loc, buf, &tot);
  if (ex < remaining && remaining <= ex + loc) {
    uint32_t cum = ex;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      if (cum + h[u] >= remaining) {
        *s_digit = (uint32_t)(1023 - 4 * tid - u);
        *s_above = cum;
        break;
      }
      cum += h[u];
    }
  }
  __syncthreads();
}

// kCluster: CTAs per row (the launch's cluster dimension).  kPerSm: CTAs the register
// budget lets one SM hold -- 5 (48 registers) for launches with more CTAs than three
// per SM hold (a prefill, a multi-token decode), so that more rows' latency chains
// overlap, else 3 (up to 80 registers: the lowest latency per row).  (Six per SM spills.)
template <int kCluster, int kPerSm = 3>
__global__ void __launch_bounds__(kThreads, kPerSm) topk_cluster_kernel(TopkParams p) {
  // candidates one CTA may put in the pool (clusters of 16 pool twice as many, so that a
  // CTA keeps 256 slots)
  constexpr int kSlot = (kCluster >= 16 ? 2 * kPoolTotal : kPoolTotal) / kCluster;
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = (int)cluster.block_rank();
  const int row = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int K = p.top_k;
  pdl_trigger();
  int b, n;  // (token metadata are inputs: read before the dependency wait)
  resolve_token(p.tv, row, &b, &n, nullptr);  // the score pass reports bad metadata
  pdl_wait();  // scores and histograms of the score kernel

  int32_t* out = p.out_idx + (int64_t)row * K;
  float* outs = p.out_score ? p.out_score + (int64_t)row * K : nullptr;
  const float* srow = p.scores + (int64_t)row * p.score_stride;

  if (n <= K) {  // every visible position is selected (uniform over the cluster)
    for (int i = rank * kThreads + tid; i < K; i += kCluster * kThreads) {
      out[i] = i < n ? i : -1;
      if (outs) outs[i] = i < n ? srow[i] : __uint_as_float(0x7FC00000u);
    }
    return;
  }

  __shared__ uint32_t cand_local[kLocalCap];
  __shared__ uint32_t pool[kCluster][kSlot];  // every CTA's candidates
  __shared__ int pool_n[kCluster], pool_above[kCluster];
  __shared__ __align__(16) uint32_t hist[1024];
  __shared__ int wcnt[kWarpsPerCta];                 // candidates each warp gathered
  __shared__ int2 wstat[2][kWarpsPerCta];            // output: each warp's #{> T}, #{== T}
  __shared__ int red[kWarpsPerCta][2 * kCluster];    // per warp: #{> T}, #{== T} of each CTA's pool
  __shared__ int buf[kWarpsPerCta];
  __shared__ int s_nlocal, s_above_local;
  __shared__ int cnt[2];  // fallback: this CTA's #{key > T}, #{key == T}
  __shared__ uint32_t s_digit, s_above;
  __shared__ int s_taken_before, s_eq_before;

  // This CTA's positions [lo, hi), visited in blocks of kBlock whose keys sit in
  // registers: warp w owns kChunks consecutive 32-position chunks of each block.
  const int chunk = ((n + kCluster - 1) / kCluster + 31) / 32 * 32;
  const int lo = min(n, rank * chunk), hi = min(n, lo + chunk);
  const int nblocks = (hi - lo + kBlock - 1) / kBlock;
  uint32_t kr[kChunks];
  auto load_block = [&](int blk) {
    const int base = lo + blk * kBlock + warp * (kChunks * 32) + lane;
#pragma unroll
    for (int c = 0; c < kChunks; ++c) {
      const int i = base + c * 32;
      kr[c] = i < hi ? score_key(__ldg(srow + i)) : 0u;
    }
  };
  // ---- 1. bin of the K-th largest key among the 4096 top-12-bit bins (all CTAs alike)
  // thread t owns bins 4095-16t .. 4080-16t (high to low); its loads go out first, the
  // CTA's first block of keys right behind them (in flight while the bins are scanned)
  const uint32_t* h12 = p.hist + (int64_t)row * kTopkBins;
  uint32_t hb[16];
  uint32_t local = 0;
  {
    const uint4* hp = (const uint4*)(h12 + kTopkBins - 16 * (tid + 1));  // this thread's 16 bins, low to high
    uint4 x[4];
#pragma unroll
    for (int v = 0; v < 4; ++v) x[v] = __ldg(hp + v);
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      hb[15 - 4 * v] = x[v].x;
      hb[14 - 4 * v] = x[v].y;
      hb[13 - 4 * v] = x[v].z;
      hb[12 - 4 * v] = x[v].w;
    }
  }
  int loaded = -1;
  if (nblocks > 0) {
    load_block(0);
    loaded = 0;
  }
#pragma unroll
  for (int u = 0; u < 16; ++u) local += hb[u];
  if (tid == 0) {
    s_nlocal = 0;
    s_above_local = 0;
    s_digit = 0;
    s_above = 0;
  }
  int tot;
  const uint32_t excl = (uint32_t)block_excl_sum((int)local, buf, &tot);
  uint32_t remaining = (uint32_t)K;
  if (excl < remaining && remaining <= excl + local) {
    uint32_t cum = excl;
    for (int u = 0; u < 16; ++u) {
      if (cum + hb[u] >= remaining) {
        s_digit = (uint32_t)(kTopkBins - 1 - 16 * tid - u);
        s_above = cum;
        break;
      }
      cum += hb[u];
    }
  }
  __syncthreads();
  const uint32_t bin = s_digit;
  uint32_t prefix = bin << 20, mask = 0xFFF00000u;
  remaining -= s_above;

  // ---- 2. this CTA's keys above the bin (counted) and in it (gathered) ---------------
  // Warp w gathers into its own slice of kLocalCap / 8 slots (no atomics); the slices
  // are concatenated when the pool is written.
  constexpr int kWarpCap = kLocalCap / kWarpsPerCta;
  {
    int above = 0, nw = 0;
    for (int blk = 0; blk < nblocks; ++blk) {
      if (loaded != blk) {
        load_block(blk);
        loaded = blk;
      }
      const int base = lo + blk * kBlock + warp * (kChunks * 32) + lane;
#pragma unroll
      for (int c = 0; c < kChunks; ++c) {
        const bool ok = base + c * 32 < hi;
        above += __popc(__ballot_sync(0xffffffffu, ok && (kr[c] >> 20) > bin));
        const bool in = ok && (kr[c] & mask) == prefix;
        const unsigned bal = __ballot_sync(0xffffffffu, in);
        const int slot = nw + __popc(bal & ((1u << lane) - 1u));
        if (in && slot < kWarpCap) cand_local[warp * kWarpCap + slot] = kr[c];
        nw += __popc(bal);
      }
    }
    if (lane == 0) {
      wcnt[warp] = nw;
      atomicAdd(&s_above_local, above);
      atomicAdd(&s_nlocal, nw);
    }
  }
  if (loaded > 0) {  // the output (or the fallback) starts over at block 0: its loads now
    load_block(0);   // overlap the pool exchange and the select
    loaded = 0;
  }
  __syncthreads();

  // ---- 3. pool (every CTA writes its part into every CTA), then one cluster barrier --
  {
    int nl = s_nlocal;
    for (int w = 0; w < kWarpsPerCta; ++w) nl = wcnt[w] > kWarpCap ? kSlot + 1 : nl;  // a full slice: fall back
    const int m = nl <= kSlot ? nl : 0;  // (an overfull CTA sends the fallback its count only)
    // entry j of the pool slot: warp slices in order
    if constexpr (kSlot <= kThreads) {
      uint32_t v = 0;
      if (tid < m) {
        int j = tid, w = 0;
        while (j >= wcnt[w]) j -= wcnt[w++];
        v = cand_local[w * kWarpCap + j];
      }
      for (int r = 0; r < kCluster; ++r) {
        uint32_t* dst = cluster.map_shared_rank(&pool[rank][0], r);
        if (tid < m) dst[tid] = v;
      }
    } else {
      for (int j0 = tid; j0 < m; j0 += kThreads) {
        int j = j0, w = 0;
        while (j >= wcnt[w]) j -= wcnt[w++];
        const uint32_t v = cand_local[w * kWarpCap + j];
        for (int r = 0; r < kCluster; ++r) *cluster.map_shared_rank(&pool[rank][j0], r) = v;
      }
    }
    if (tid < kCluster) {
      *cluster.map_shared_rank(&pool_n[rank], tid) = nl;
      *cluster.map_shared_rank(&pool_above[rank], tid) = s_above_local;
    }
  }
  cluster.sync();
  bool fast = true;
  for (int r = 0; r < kCluster; ++r) fast = fast && pool_n[r] <= kSlot;

  const unsigned lt = (1u << lane) - 1u;
  int taken0, ties0;  // this CTA's first output slot and #{key == T} before it
  uint32_t T;
  if (fast) {
    // exact K-th largest key among the pooled candidates (all keys of the bin): MSB-first
    // radix select over the remaining 20 bits, 10 at a time
#pragma unroll 1
    for (int pass = 0; pass < 2; ++pass) {
      const int shift = pass == 0 ? 10 : 0;
      const uint32_t dmask = 0x3FFu;
#pragma unroll
      for (int u = 0; u < 1024 / kThreads; ++u) hist[tid + u * kThreads] = 0;
      __syncthreads();
      if constexpr (kSlot <= kThreads) {  // one pool entry per thread and CTA
#pragma unroll
        for (int r = 0; r < kCluster; ++r)
          if (tid < pool_n[r]) {
            const uint32_t k = pool[r][tid];
            if ((k & mask) == prefix) atomicAdd(&hist[(k >> shift) & dmask], 1u);
          }
      } else {
        for (int r = 0; r < kCluster; ++r)
          for (int j = tid; j < pool_n[r]; j += kThreads) {
            const uint32_t k = pool[r][j];
            if ((k & mask) == prefix) atomicAdd(&hist[(k >> shift) & dmask], 1u);
          }
      }
      __syncthreads();
      find_bin1024(hist, remaining, buf, &s_digit, &s_above);
      prefix |= s_digit << shift;
      mask |= dmask << shift;
      remaining -= s_above;
    }
    T = prefix;  // take `remaining` of the keys == T
    // #{> T} and #{== T} in every CTA's pool: counted per thread, summed over each warp
    // and then over the warps
    {
#pragma unroll
      for (int r = 0; r < kCluster; ++r) {
        int g, e;
        if constexpr (kSlot <= kThreads) {
          const bool has = tid < pool_n[r];
          const uint32_t k = has ? pool[r][tid] : 0u;
          g = __popc(__ballot_sync(0xffffffffu, has && k > T));
          e = __popc(__ballot_sync(0xffffffffu, has && k == T));
        } else {
          g = 0;
          e = 0;
          for (int j = tid; j < pool_n[r]; j += kThreads) {
            const uint32_t k = pool[r][j];
            g += k > T;
            e += k == T;
          }
          g = __reduce_add_sync(0xffffffffu, g);
          e = __reduce_add_sync(0xffffffffu, e);
        }
        if (lane == 0) {
          red[warp][r] = g;
          red[warp][kCluster + r] = e;
        }
      }
    }
    __syncthreads();
    // place this CTA after the ones before it (warp 0; lane r < kCluster speaks for CTA r)
    if (warp == 0) {
      int gt_r = 0, eq_r = 0;
      if (lane < kCluster) {
        gt_r = pool_above[lane];
#pragma unroll
        for (int w = 0; w < kWarpsPerCta; ++w) {
          gt_r += red[w][lane];
          eq_r += red[w][kCluster + lane];
        }
      }
      int taken = 0, eq_before = 0;
      for (int r = 0; r < rank; ++r) {  // the whole warp, in step
        const int g = __shfl_sync(0xffffffffu, gt_r, r);
        const int e = __shfl_sync(0xffffffffu, eq_r, r);
        taken += g + max(0, min((int)remaining - eq_before, e));
        eq_before += e;
      }
      if (lane == 0) {
        s_taken_before = taken;
        s_eq_before = eq_before;
      }
    }
    __syncthreads();
    taken0 = s_taken_before;
    ties0 = s_eq_before;
  } else {
    // fallback: an MSB-first radix select over the remaining 20 bits (8 + 8 + 4): each
    // CTA counts its own keys (the row's r-th C-th, from registers) into a 256-bin
    // histogram, and the cluster sums the CTAs' histograms through distributed shared
    // memory (one barrier once all are counted, one once all are read, since the next
    // pass recounts into the same bins); counts are exchanged the same way below
#pragma unroll 1
    for (int pass = 0; pass < 3; ++pass) {
      const int shift = pass == 0 ? 12 : (pass == 1 ? 4 : 0);
      const uint32_t dmask = pass == 2 ? 0xFu : 0xFFu;
      hist[tid] = 0;
      __syncthreads();
      for (int blk = 0; blk < nblocks; ++blk) {
        if (loaded != blk) {
          load_block(blk);
          loaded = blk;
        }
        const int base = lo + blk * kBlock + warp * (kChunks * 32) + lane;
#pragma unroll
        for (int c = 0; c < kChunks; ++c) {
          const uint32_t k = kr[c];
          const bool in = base + c * 32 < hi && (k & mask) == prefix;
          const unsigned act = __ballot_sync(0xffffffffu, in);
          if (in) {
            const unsigned peers = __match_any_sync(act, (k >> shift) & dmask);
            if (lane == __ffs(peers) - 1) atomicAdd(&hist[(k >> shift) & dmask], (uint32_t)__popc(peers));
          }
        }
      }
      __syncthreads();
      cluster.sync();  // every CTA's counts are in its hist[0, 256)
      uint32_t tot = 0;
      for (int r = 0; r < kCluster; ++r) tot += *cluster.map_shared_rank(&hist[tid], r);
      cluster.sync();  // every CTA has read them (the next pass recounts into them)
      hist[256 + tid] = tot;
      __syncthreads();
      if (warp == 0) find_bin256(hist + 256, remaining, &s_digit, &s_above);
      __syncthreads();
      prefix |= s_digit << shift;
      mask |= dmask << shift;
      remaining -= s_above;
    }
    T = prefix;
    int gt_c = 0, eq_c = 0;
    for (int blk = 0; blk < nblocks; ++blk) {
      if (loaded != blk) {
        load_block(blk);
        loaded = blk;
      }
      const int base = lo + blk * kBlock + warp * (kChunks * 32) + lane;
#pragma unroll
      for (int c = 0; c < kChunks; ++c) {
        const bool ok = base + c * 32 < hi;
        gt_c += (ok && kr[c] > T);
        eq_c += (ok && kr[c] == T);
      }
    }
    for (int o = 16; o; o >>= 1) {
      gt_c += __shfl_xor_sync(0xffffffffu, gt_c, o);
      eq_c += __shfl_xor_sync(0xffffffffu, eq_c, o);
    }
    if (tid == 0) cnt[0] = cnt[1] = 0;
    __syncthreads();
    if (lane == 0) {
      atomicAdd(&cnt[0], gt_c);
      atomicAdd(&cnt[1], eq_c);
    }
    cluster.sync();
    if (tid == 0) {
      int taken = 0, eq_before = 0;
      for (int r = 0; r < rank; ++r) {
        const int* c = cluster.map_shared_rank(cnt, r);
        taken += c[0] + max(0, min((int)remaining - eq_before, c[1]));
        eq_before += c[1];
      }
      s_taken_before = taken;
      s_eq_before = eq_before;
    }
    cluster.sync();  // no CTA leaves while another may still read its shared memory
    taken0 = s_taken_before;
    ties0 = s_eq_before;
  }

  // ---- 4. ordered output -------------------------------------------------------------
  int taken = taken0, ties = ties0;  // before the current block
  for (int blk = 0; blk < nblocks; ++blk) {
    if (loaded != blk) {
      load_block(blk);
      loaded = blk;
    }
    const int base = lo + blk * kBlock + warp * (kChunks * 32) + lane;
    int gt_w = 0, eq_w = 0;
#pragma unroll
    for (int c = 0; c < kChunks; ++c) {
      const bool ok = base + c * 32 < hi;
      gt_w += __popc(__ballot_sync(0xffffffffu, ok && kr[c] > T));
      eq_w += __popc(__ballot_sync(0xffffffffu, ok && kr[c] == T));
    }
    // every warp publishes its counts (double-buffered over blocks: one barrier each);
    // each warp then places itself after the warps before it and sums the block
    if (lane == 0) wstat[blk & 1][warp] = make_int2(gt_w, eq_w);
    __syncthreads();
    int eq_before = ties, pos = taken, eq_tot = 0, tk_tot = 0;
#pragma unroll
    for (int w = 0; w < kWarpsPerCta; ++w) {
      const int2 st = wstat[blk & 1][w];
      const int tk = st.x + max(0, min((int)remaining - (ties + eq_tot), st.y));
      if (w < warp) {
        eq_before += st.y;
        pos += tk;
      }
      eq_tot += st.y;
      tk_tot += tk;
    }
    int tie = eq_before;
#pragma unroll
    for (int c = 0; c < kChunks; ++c) {
      const bool ok = base + c * 32 < hi;
      const bool gt = ok && kr[c] > T;
      const bool eq = ok && kr[c] == T;
      const unsigned eqb = __ballot_sync(0xffffffffu, eq);
      const bool take = gt || (eq && tie + __popc(eqb & lt) < (int)remaining);
      const unsigned tkb = __ballot_sync(0xffffffffu, take);
      const int dst = pos + __popc(tkb & lt);
      if (take && dst < K) {
        out[dst] = base + c * 32;
        if (outs) outs[dst] = key_score(kr[c]);
      }
      pos += __popc(tkb);
      tie += __popc(eqb);
    }
    taken += tk_tot;
    ties += eq_tot;
  }
}

}  // namespace

cudaError_t launch_topk(const TopkParams& p, int32_t max_visible, cudaStream_t s) {
  // the fewest CTAs per row that keep each CTA's share of the longest row within one
  // block of keys held in registers (more for longer rows: 16, a non-portable cluster
  // size, beyond 8 blocks; where a device cannot run clusters of 16, 8)
  const int cl = max_visible <= kBlock ? 1 : max_visible <= 2 * kBlock ? 2 : max_visible <= 4 * kBlock ? 4
               : max_visible <= 8 * kBlock ? 8 : 16;
  const dim3 b(kThreads);
  // more rows than three CTAs per SM hold at once: the five-per-SM variant
  const bool many = (int64_t)p.tv.n_tokens * cl > 3 * (int64_t)device_sm_count();
  switch (cl) {
    case 1:
      return many ? launch_pdl_cluster(topk_cluster_kernel<1, 5>, dim3(1, p.tv.n_tokens), b, 0, s, 1u, p)
                  : launch_pdl_cluster(topk_cluster_kernel<1>, dim3(1, p.tv.n_tokens), b, 0, s, 1u, p);
    case 2:
      return many ? launch_pdl_cluster(topk_cluster_kernel<2, 5>, dim3(2, p.tv.n_tokens), b, 0, s, 2u, p)
                  : launch_pdl_cluster(topk_cluster_kernel<2>, dim3(2, p.tv.n_tokens), b, 0, s, 2u, p);
    case 4:
      return many ? launch_pdl_cluster(topk_cluster_kernel<4, 5>, dim3(4, p.tv.n_tokens), b, 0, s, 4u, p)
                  : launch_pdl_cluster(topk_cluster_kernel<4>, dim3(4, p.tv.n_tokens), b, 0, s, 4u, p);
    case 8:
      return many ? launch_pdl_cluster(topk_cluster_kernel<8, 5>, dim3(8, p.tv.n_tokens), b, 0, s, 8u, p)
                  : launch_pdl_cluster(topk_cluster_kernel<8>, dim3(8, p.tv.n_tokens), b, 0, s, 8u, p);
    default: {
      static std::atomic<int> allowed[kMaxDevices];  // 1: set, -1: refused on that device
      int dev = 0;
      cudaError_t e = cudaGetDevice(&dev);
      if (e != cudaSuccess) return e;
      const int idx = dev >= 0 && dev < kMaxDevices ? dev : 0;
      if (allowed[idx].load(std::memory_order_acquire) == 0) {
        e = cudaFuncSetAttribute(topk_cluster_kernel<16>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        allowed[idx].store(e == cudaSuccess ? 1 : -1, std::memory_order_release);
        if (e != cudaSuccess) (void)cudaGetLastError();
      }
      if (allowed[idx].load(std::memory_order_acquire) == 1) {
        e = launch_pdl_cluster(topk_cluster_kernel<16>, dim3(16, p.tv.n_tokens), b, 0, s, 16u, p);
        if (e == cudaSuccess) return e;
        (void)cudaGetLastError();  // a device without room for clusters of 16: eight CTAs per row
      }
      return launch_pdl_cluster(topk_cluster_kernel<8>, dim3(8, p.tv.n_tokens), b, 0, s, 8u, p);
    }
  }
}

}  // namespace dsa
