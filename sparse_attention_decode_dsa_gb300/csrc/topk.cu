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
// top 12 bits (kept in the workspace).  One CTA per row then
//   1. finds the bin holding the K-th largest key from that histogram;
//   2. gathers the keys of that bin (the candidates) into shared memory;
//   3. finds the exact K-th largest key T among them with an MSB-first radix select
//      over the remaining 20 bits (8 + 8 + 4), and how many keys equal to T to take;
//   4. writes, in position order, every key > T and the first (K - #{> T}) keys == T:
//      each warp owns contiguous ranges; a count, a block scan that places the warps,
//      and a write.
// Keys are read from the score row in blocks of 32768 positions held in registers (32
// per thread, all loads issued together), so a row of up to 32768 positions is read
// from L2 once.
// If the candidates overflow shared memory (a row with very many equal top bits), step
// 3 scans the whole row instead of the candidate list, with the same result.
#include "common.cuh"

namespace dsa {

namespace {

constexpr int kTopkThreads = 1024;
constexpr int kCandCap = 24576;  // candidate keys kept in shared memory
constexpr int kChunks = 32;                          // 32-position chunks per warp per block
constexpr int kBlock = kTopkThreads * kChunks;       // positions whose keys sit in registers

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
  if (warp == 0) {
    const int c = buf[lane];  // 32 warps
    int s = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += u;
    }
    buf[lane] = s - c;            // exclusive prefix of the warp totals
    if (lane == 31) buf[32] = s;  // CTA total
  }
  __syncthreads();
  const int before = buf[warp];
  *total = buf[32];
  __syncthreads();  // buf is reused by the next call
  return before + incl - v;
}

__global__ void __launch_bounds__(kTopkThreads) topk_row_kernel(TopkParams p) {
  const int row = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int K = p.top_k;

  int b, n;
  resolve_token(p.tv, row, &b, &n, nullptr);  // the score pass reports bad metadata
  int32_t* out = p.out_idx + (int64_t)row * K;
  float* outs = p.out_score ? p.out_score + (int64_t)row * K : nullptr;
  const float* srow = p.scores + (int64_t)row * p.score_stride;

  if (n <= K) {  // every visible position is selected
    for (int i = tid; i < K; i += kTopkThreads) {
      out[i] = i < n ? i : -1;
      if (outs) outs[i] = i < n ? srow[i] : __uint_as_float(0x7FC00000u);
    }
    return;
  }

  extern __shared__ uint32_t cand[];  // [kCandCap] keys of the boundary bin
  __shared__ int buf[33];
  __shared__ uint32_t hist[256];
  __shared__ uint32_t s_digit, s_above;
  __shared__ int s_ncand;

  // ---- 1. bin of the K-th largest key among the 4096 top-12-bit bins ----------------
  // thread t owns bins 4095-4t .. 4092-4t (high to low)
  const uint32_t* h12 = p.hist + (int64_t)row * kTopkBins;
  uint32_t hb[4];
  uint32_t local = 0;
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    hb[u] = __ldg(h12 + kTopkBins - 1 - 4 * tid - u);
    local += hb[u];
  }
  if (tid == 0) {
    s_ncand = 0;
    s_digit = 0;
    s_above = 0;
  }
  int tot;
  const uint32_t excl = (uint32_t)block_excl_sum((int)local, buf, &tot);
  uint32_t remaining = (uint32_t)K;
  if (excl < remaining && remaining <= excl + local) {
    uint32_t cum = excl;
    for (int u = 0; u < 4; ++u) {
      if (cum + hb[u] >= remaining) {
        s_digit = (uint32_t)(kTopkBins - 1 - 4 * tid - u);
        s_above = cum;
        break;
      }
      cum += hb[u];
    }
  }
  __syncthreads();
  uint32_t prefix = s_digit << 20, mask = 0xFFF00000u;
  remaining -= s_above;

  // Positions are visited in blocks of kBlock; within a block warp w owns the kChunks
  // consecutive 32-position chunks starting at w * kChunks * 32, lane l the l-th of each.
  // A block's keys are loaded into registers with all loads in flight at once.
  const int nblocks = (n + kBlock - 1) / kBlock;
  uint32_t kr[kChunks];
  auto load_block = [&](int blk) {
    const int base = blk * kBlock + warp * (kChunks * 32) + lane;
#pragma unroll
    for (int c = 0; c < kChunks; ++c) {
      const int i = base + c * 32;
      kr[c] = i < n ? score_key(__ldg(srow + i)) : 0u;
    }
  };
  int loaded = -1;

  // ---- 2. gather the keys of that bin ---------------------------------------------
  for (int blk = 0; blk < nblocks; ++blk) {
    load_block(blk);
    loaded = blk;
    const int base = blk * kBlock + warp * (kChunks * 32) + lane;
#pragma unroll
    for (int c = 0; c < kChunks; ++c) {
      const bool in = base + c * 32 < n && (kr[c] & mask) == prefix;
      const unsigned bal = __ballot_sync(0xffffffffu, in);
      if (bal) {
        int slot = 0;
        if (lane == 0) slot = atomicAdd(&s_ncand, __popc(bal));
        slot = __shfl_sync(0xffffffffu, slot, 0) + __popc(bal & ((1u << lane) - 1u));
        if (in && slot < kCandCap) cand[slot] = kr[c];
      }
    }
  }
  __syncthreads();
  const int ncand = s_ncand;
  const bool use_cand = ncand <= kCandCap;

  // ---- 3. exact K-th largest key: radix select over the low 20 bits ---------------
#pragma unroll 1
  for (int pass = 0; pass < 3; ++pass) {
    const int shift = pass == 0 ? 12 : (pass == 1 ? 4 : 0);
    const uint32_t dmask = pass == 2 ? 0xFu : 0xFFu;
    if (tid < 256) hist[tid] = 0;
    __syncthreads();
    const int cnt = use_cand ? ncand : n;
    for (int base = 0; base < cnt; base += kTopkThreads) {
      const int i = base + tid;
      uint32_t k = 0;
      if (i < cnt) k = use_cand ? cand[i] : score_key(srow[i]);
      const bool in = i < cnt && (k & mask) == prefix;
      const uint32_t dgt = (k >> shift) & dmask;
      const unsigned act = __ballot_sync(0xffffffffu, in);
      if (in) {
        const unsigned peers = __match_any_sync(act, dgt);
        if (lane == __ffs(peers) - 1) atomicAdd(&hist[dgt], (uint32_t)__popc(peers));
      }
    }
    __syncthreads();
    if (warp == 0) {
      // lane l owns bins 255-8l .. 248-8l (high to low)
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
            s_digit = (uint32_t)bin;
            s_above = cum;
            break;
          }
          cum += hist[bin];
        }
      }
    }
    __syncthreads();
    prefix |= s_digit << shift;
    mask |= dmask << shift;
    remaining -= s_above;
  }
  const uint32_t T = prefix;  // the K-th largest key; take `remaining` of the keys == T

  // ---- 4. ordered output, block by block ---------------------------------------------
  const unsigned lt = (1u << lane) - 1u;
  int taken = 0, ties = 0;  // row-wide, before the current block
  for (int blk = 0; blk < nblocks; ++blk) {
    if (loaded != blk) {
      load_block(blk);
      loaded = blk;
    }
    const int base = blk * kBlock + warp * (kChunks * 32) + lane;
    int gt_w = 0, eq_w = 0;
#pragma unroll
    for (int c = 0; c < kChunks; ++c) {
      const bool ok = base + c * 32 < n;
      gt_w += __popc(__ballot_sync(0xffffffffu, ok && kr[c] > T));
      eq_w += __popc(__ballot_sync(0xffffffffu, ok && kr[c] == T));
    }
    int eq_tot;
    // every lane of a warp holds the warp's counts; lane 0 alone enters them in the scans
    const int eq_before = ties + __shfl_sync(0xffffffffu, block_excl_sum(lane == 0 ? eq_w : 0, buf, &eq_tot), 0);
    const int take_w = gt_w + max(0, min((int)remaining - eq_before, eq_w));
    int tk_tot;
    int pos = taken + __shfl_sync(0xffffffffu, block_excl_sum(lane == 0 ? take_w : 0, buf, &tk_tot), 0);
    int tie = eq_before;
#pragma unroll
    for (int c = 0; c < kChunks; ++c) {
      const bool ok = base + c * 32 < n;
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
  (void)max_visible;
  const size_t smem = (size_t)kCandCap * sizeof(uint32_t);
  cudaError_t e = cudaFuncSetAttribute(topk_row_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  topk_row_kernel<<<p.tv.n_tokens, kTopkThreads, smem, s>>>(p);
  return cudaGetLastError();
}

}  // namespace dsa
