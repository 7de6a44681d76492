// Sparse Flash Attention on the 5th-generation tensor cores (tcgen05), one CTA pair per
// (query token, split of its index list).
//
// "Adapting and Optimizing Inference for a New Model Architecture on Ascend", section
// 3.1: attention over only the selected Top-K positions, read from the main-attention
// KV cache by index; "Inference Acceleration for Next-Gen Attention Architectures",
// section 3.2: the rows are non-contiguous, fetched by paged addressing.  DSA builds on
// MLA ("Day0 Inference Optimization on Ascend CANN", section 1): every head attends over
// the same 576-wide latent row, whose leading 512 entries are the value.
//
// Work split inside the pair (CTA c = 0, 1):
//   * CTA c owns value dims [256c, 256c + 256) of the output, and contracts the logits
//     over its 288 "own" dims: latent [256c, 256c + 256) and rope [512 + 32c, +32), so
//     each CTA gathers exactly half of every selected 1152-byte row.
//   * Each CTA computes partial logits S_c = Q[:, own] . KV[:, own]^T (tcgen05, A = Q
//     from tensor memory, B = gathered rows in shared memory), sends them to its peer
//     through distributed shared memory (st.async, counted on the peer's mbarrier) and
//     adds the peer's part: both CTAs hold the same S = S_0 + S_1.
//   * Online softmax per head row (thread = row, no shuffles), base 2; the reference
//     maximum only moves when a tile's maximum exceeds it by 8 (2^8 headroom), and O is
//     then rescaled in tensor memory.
//   * P (bf16) goes to tensor memory; O[128 x 256] += P . V with V read MN-major from
//     the same shared-memory rows the logits used.
// Warp roles: warp 0 gathers rows with 16-byte cp.async into a 4-stage ring laid out in
// 128-byte swizzle atoms; warp 1 (one thread) issues the MMAs; warps 2-5 run softmax
// and the epilogue.  Tensor memory (512 columns): O [0,256), S [256,320), P [320,352),
// Q rope [352,368), Q latent [384,512).  Every wait is bounded.
#include "sm100.cuh"

namespace dsa {

namespace {

using namespace sm100;

constexpr int kThreads = 192;
constexpr int kTok = 64;                         // selected positions per tile
constexpr int kStages = 4;
constexpr int kRegion = kTok * 128;              // 64 rows x 128 B
constexpr int kStageBytes = 5 * kRegion;         // 4 latent regions + 1 rope region
constexpr int kXchBytes = 128 * kTok * 4;        // one f32 partial-logit tile
constexpr int kMaxSplitLen = kMaxTopK;
constexpr uint32_t kColO = 0, kColS = 256, kColP = 320, kColQr = 352, kColQl = 384;
constexpr int kSmem = 1024 + kStages * kStageBytes + kXchBytes + kMaxSplitLen * 4 + 512;

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1) sfa_tc_kernel(SfaParams p) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t c = cluster_rank();
  const uint32_t peer = c ^ 1u;
  const int split = blockIdx.x >> 1, tok = blockIdx.y;
  const int H = p.n_heads;

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u32 = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024 - (raw_u32 & 1023)) & 1023);
  uint8_t* stages = smem;
  float* xch = (float*)(stages + kStages * kStageBytes);      // [128 rows][64] peer partial
  int32_t* rowid = (int32_t*)((uint8_t*)xch + kXchBytes);     // cache row of each slot or -1
  uint64_t* bars = (uint64_t*)(rowid + kMaxSplitLen);
  uint64_t* kv_full = bars;
  uint64_t* kv_empty = kv_full + kStages;
  uint64_t* q_ready = kv_empty + kStages;
  uint64_t* s_full = q_ready + 1;
  uint64_t* s_free = s_full + 1;
  uint64_t* p_full = s_free + 1;
  uint64_t* pv_done = p_full + 1;
  uint64_t* xch_full = pv_done + 1;
  uint64_t* xch_empty = xch_full + 1;
  uint64_t* drain = xch_empty + 1;
  uint32_t* tmem_base_s = (uint32_t*)(drain + 1);
  volatile int* abort_flag = (volatile int*)(tmem_base_s + 1);

  int b, n_vis;
  resolve_token(p.tv, tok, &b, &n_vis, nullptr);
  const int j_begin = split * p.split_len;
  const int j_end = min(p.top_k, j_begin + p.split_len);
  const int ntok = max(0, j_end - j_begin);
  const int n_tiles = (ntok + kTok - 1) / kTok;

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&kv_full[s], 1);
      mbar_init(&kv_empty[s], 1);
    }
    mbar_init(q_ready, 4);
    mbar_init(s_full, 1);
    mbar_init(s_free, 4);
    mbar_init(p_full, 4);
    mbar_init(pv_done, 1);
    mbar_init(xch_full, 1);
    mbar_init(xch_empty, 4);  // the peer's four softmax warps
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
    if (n_tiles > 0) mbar_arrive_expect_tx(xch_full, kXchBytes);  // the peer's tile-0 partial
  }
  if (warp == 1) {
    tmem_alloc(tmem_base_s, 512);
    tmem_relinquish();
  }
  // cache rows of the selected positions of this split (-1: padding or invalid)
  for (int j = tid; j < n_tiles * kTok; j += kThreads) {
    const int jj = j_begin + j;
    int rid = -1;
    if (jj < j_end) {
      const int pos = __ldg(p.idx + (int64_t)tok * p.top_k + jj);
      if (pos >= n_vis || pos < -1) {
        if (c == 0) atomicOr(p.err, DSA_DEVERR_INDEX);
      } else if (pos >= 0) {
        const int pg = physical_page(p.tv, b, pos >> 6, c == 0 ? p.err : nullptr);
        if (pg >= 0) rid = pg * kPage + (pos & 63);
      }
    }
    rowid[j] = rid;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  cluster_sync_all();  // both CTAs' barriers exist before any remote traffic
  const uint32_t tmem = *tmem_base_s;

  if (warp == 0) {
    // ============================ gather (cp.async) ====================================
    // Tile n's copies are known complete (cp.async.wait_group) when tile n + kLag has
    // been issued; only then is it signalled.  Before the producer blocks on a stage
    // (tile n needs the stage of tile n - kStages, freed by P.V of that tile, which the
    // MMA issues after the logits of tile n - kStages + 1), that tile must already be
    // signalled: n - 1 - kLag >= n - kStages + 1, i.e. kLag <= kStages - 2.
    constexpr int kLag = kStages - 2;
    const uint16_t* kv = p.kv;
    int n = 0, signalled = 0;
    for (; n < n_tiles; ++n) {
      const int stage = n % kStages;
      bool ok = true;
      if (lane == 0) ok = mbar_wait(&kv_empty[stage], ((n / kStages) & 1) ^ 1, abort_flag, p.err);
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      const uint32_t sbase = smem_u32(stages + stage * kStageBytes);
#pragma unroll
      for (int rr = 0; rr < 2; ++rr) {
        const int j = lane + 32 * rr;
        const int rid = rowid[n * kTok + j];
        const int bytes = rid >= 0 ? 16 : 0;
        const uint16_t* src = kv + (int64_t)(rid >= 0 ? rid : 0) * kLatentDim;
        const uint32_t rowbase = sbase + j * 128;
        const uint32_t sw = (uint32_t)(j & 7);
#pragma unroll
        for (int u = 0; u < 32; ++u) {  // own latent dims: 4 regions x 8 chunks of 16 B
          cp_async_16(rowbase + (u >> 3) * kRegion + ((((uint32_t)u & 7u) ^ sw) << 4), src + 256 * c + u * 8, bytes);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {  // own rope dims: first 64 B of the rope region row
          cp_async_16(rowbase + 4 * kRegion + (((uint32_t)u ^ sw) << 4), src + 512 + 32 * c + u * 8, bytes);
        }
      }
      cp_async_commit();
      if (n >= kLag) {
        cp_async_wait<kLag>();
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&kv_full[(n - kLag) % kStages]);
        signalled = n - kLag + 1;
      }
    }
    cp_async_wait<0>();
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0 && !*abort_flag) {
      for (int m = signalled; m < n; ++m) mbar_arrive(&kv_full[m % kStages]);
    }
  } else if (warp == 1) {
    // ============================ MMA issuer ==========================================
    if (lane == 0) {
      const uint32_t id_qk = idesc(128, kTok, 1u, 1u);
      const uint32_t id_pv = idesc_bmn(128, 256, 1u, 1u);
      bool ok = mbar_wait(q_ready, 0, abort_flag, p.err);
      for (int n = 0; ok && n <= n_tiles; ++n) {
        if (n < n_tiles) {
          const int stage = n % kStages;
          if (!(ok = mbar_wait(&kv_full[stage], (n / kStages) & 1, abort_flag, p.err))) break;
          if (n > 0 && !(ok = mbar_wait(s_free, (n - 1) & 1, abort_flag, p.err))) break;
          tc_fence_after();
          const uint32_t sb = smem_u32(stages + stage * kStageBytes);
#pragma unroll
          for (int k = 0; k < 18; ++k) {  // 16 latent steps + 2 rope steps of 16 dims
            const uint32_t a = tmem + (k < 16 ? kColQl + 8 * k : kColQr + 8 * (k - 16));
            const uint32_t boff = k < 16 ? (k >> 2) * kRegion + (k & 3) * 32 : 4 * kRegion + (k - 16) * 32;
            mma_f16_ts(tmem + kColS, a, desc_sw128(sb + boff), id_qk, k > 0);
          }
          tc_commit(s_full);
        }
        if (n > 0) {
          const int m = n - 1, stage = m % kStages;
          if (!(ok = mbar_wait(p_full, m & 1, abort_flag, p.err))) break;
          tc_fence_after();
          const uint32_t sb = smem_u32(stages + stage * kStageBytes);
#pragma unroll
          for (int j = 0; j < kTok / 16; ++j)
            mma_f16_ts(tmem + kColO, tmem + kColP + 8 * j, desc_sw128_mn(sb + j * 2048, kRegion, 1024), id_pv,
                       (m > 0 || j > 0) ? 1u : 0u);
          tc_commit(pv_done);
          tc_commit(&kv_empty[stage]);
        }
      }
      tc_commit(drain);
      const long long t0 = clock64();
      while (!mbar_try_wait(smem_u32(drain), 0) && clock64() - t0 < kWaitLimitCycles) {
      }
    }
  } else {
    // ============================ softmax + epilogue ==================================
    const int quarter = warp & 3;
    const int h = quarter * 32 + lane;  // head row == TMEM lane
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    // Q (own dims) into tensor memory as packed bf16 pairs
    {
      const bool live = h < H;
      const uint4* q4 = (const uint4*)(p.q + ((int64_t)tok * H + (live ? h : 0)) * kLatentDim);
#pragma unroll 1
      for (int ch = 0; ch < 4; ++ch) {  // latent: 4 x 32 columns (64 dims each)
        uint32_t w[32];
#pragma unroll
        for (int v = 0; v < 8; ++v) {
          const uint4 x = live ? __ldg(q4 + (256 * c + 64 * ch) / 8 + v) : make_uint4(0, 0, 0, 0);
          w[4 * v] = x.x;
          w[4 * v + 1] = x.y;
          w[4 * v + 2] = x.z;
          w[4 * v + 3] = x.w;
        }
        tmem_st32(tmem + lane_off + kColQl + 32 * ch, w);
      }
      uint32_t wr[16];
#pragma unroll
      for (int v = 0; v < 4; ++v) {
        const uint4 x = live ? __ldg(q4 + (512 + 32 * c) / 8 + v) : make_uint4(0, 0, 0, 0);
        wr[4 * v] = x.x;
        wr[4 * v + 1] = x.y;
        wr[4 * v + 2] = x.z;
        wr[4 * v + 3] = x.w;
      }
      tmem_st16(tmem + lane_off + kColQr, wr);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(q_ready);
    }
    const uint32_t xch_local = smem_u32(xch);
    const uint32_t xch_peer = map_to_rank(xch_local, peer);
    const uint32_t xfull_peer = map_to_rank(smem_u32(xch_full), peer);
    const uint32_t xempty_peer = map_to_rank(smem_u32(xch_empty), peer);
    const uint32_t myrow = (uint32_t)h * (kTok * 4);
    const uint32_t sw = (uint32_t)(h & 7);
    float m_ref = -INFINITY, l = 0.f;
    bool ok = true;
    for (int n = 0; n < n_tiles; ++n) {
      if (lane == 0) ok = mbar_wait(s_full, n & 1, abort_flag, p.err);
      if (!__shfl_sync(0xffffffffu, ok, 0)) { ok = false; break; }
      tc_fence_after();
      float s[kTok];
      {
        uint32_t v0[32], v1[32];
        tmem_ld32(tmem + lane_off + kColS, v0);
        tmem_ld32(tmem + lane_off + kColS + 32, v1);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          s[j] = __uint_as_float(v0[j]);
          s[32 + j] = __uint_as_float(v1[j]);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(s_free);
      // exchange partial logits with the peer
      if (n > 0) {
        if (lane == 0) ok = mbar_wait(xch_empty, (n - 1) & 1, abort_flag, p.err);
        if (!__shfl_sync(0xffffffffu, ok, 0)) { ok = false; break; }
      }
#pragma unroll
      for (int u = 0; u < kTok / 4; ++u)
        st_async_v4(xch_peer + myrow + (((uint32_t)u ^ sw) << 4),
                    make_float4(s[4 * u], s[4 * u + 1], s[4 * u + 2], s[4 * u + 3]), xfull_peer);
      if (lane == 0) ok = mbar_wait(xch_full, n & 1, abort_flag, p.err);
      if (!__shfl_sync(0xffffffffu, ok, 0)) { ok = false; break; }
      if (h == 0 && n + 1 < n_tiles) mbar_arrive_expect_tx(xch_full, kXchBytes);  // next tile's partial
#pragma unroll
      for (int u = 0; u < kTok / 4; ++u) {
        const float4 r = *(const float4*)((const uint8_t*)xch + myrow + (((uint32_t)u ^ sw) << 4));
        s[4 * u] += r.x;
        s[4 * u + 1] += r.y;
        s[4 * u + 2] += r.z;
        s[4 * u + 3] += r.w;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive_remote(xempty_peer);
      // online softmax (base 2), masked positions get no weight
      const int32_t* rt = rowid + n * kTok;
      float tmax = -INFINITY;
#pragma unroll
      for (int j = 0; j < kTok; ++j) {
        s[j] = rt[j] >= 0 ? s[j] * p.scale_log2 : -INFINITY;
        tmax = fmaxf(tmax, s[j]);
      }
      float alpha = 1.f;
      bool rescale = false;
      if (tmax != -INFINITY && (m_ref == -INFINITY || tmax > m_ref + 8.f)) {
        if (m_ref != -INFINITY) {
          alpha = exp2f(m_ref - tmax);
          rescale = true;
        }
        m_ref = tmax;
      }
      float rs = 0.f;
      const float msub = m_ref == -INFINITY ? 0.f : m_ref;  // nothing visible yet: all weights 0
#pragma unroll
      for (int j = 0; j < kTok; ++j) {
        s[j] = exp2f(s[j] - msub);  // exp2(-inf) = 0 for masked positions
        rs += s[j];
      }
      l = l * alpha + rs;
      if (n > 0) {
        if (lane == 0) ok = mbar_wait(pv_done, (n - 1) & 1, abort_flag, p.err);
        if (!__shfl_sync(0xffffffffu, ok, 0)) { ok = false; break; }
        tc_fence_after();
      }
      if (__any_sync(0xffffffffu, rescale)) {  // rare: move O to the new reference maximum
#pragma unroll 1
        for (int ch = 0; ch < 8; ++ch) {
          uint32_t v[32];
          tmem_ld32(tmem + lane_off + kColO + 32 * ch, v);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] = __float_as_uint(__uint_as_float(v[j]) * alpha);
          tmem_st32(tmem + lane_off + kColO + 32 * ch, v);
        }
      }
      {
        uint32_t pw[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) pw[j] = pack_bf16x2(s[2 * j], s[2 * j + 1]);
        tmem_st32(tmem + lane_off + kColP, pw);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full);
    }
    // ---- epilogue: O / l -> this CTA's 256 value dims ----------------------------------
    if (ok && n_tiles > 0) {
      if (lane == 0) ok = mbar_wait(pv_done, (n_tiles - 1) & 1, abort_flag, p.err);
      ok = __shfl_sync(0xffffffffu, ok, 0);
    }
    if (ok) {
      tc_fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      const bool live = h < H;
#pragma unroll 1
      for (int ch = 0; ch < 8; ++ch) {
        uint32_t v[32];
        if (n_tiles > 0) {
          tmem_ld32(tmem + lane_off + kColO + 32 * ch, v);
          tmem_ld_wait();
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] = 0u;
        }
        if (!live) continue;
        const int d0 = 256 * (int)c + 32 * ch;
        if (p.n_splits == 1) {
          uint4* dst = (uint4*)(p.out + ((int64_t)tok * H + h) * kValueDim + d0);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint4 w;
            w.x = pack_bf16x2(__uint_as_float(v[8 * q]) * inv, __uint_as_float(v[8 * q + 1]) * inv);
            w.y = pack_bf16x2(__uint_as_float(v[8 * q + 2]) * inv, __uint_as_float(v[8 * q + 3]) * inv);
            w.z = pack_bf16x2(__uint_as_float(v[8 * q + 4]) * inv, __uint_as_float(v[8 * q + 5]) * inv);
            w.w = pack_bf16x2(__uint_as_float(v[8 * q + 6]) * inv, __uint_as_float(v[8 * q + 7]) * inv);
            dst[q] = w;
          }
        } else {
          float4* dst = (float4*)(p.part_o + (((int64_t)tok * p.n_splits + split) * H + h) * kValueDim + d0);
#pragma unroll
          for (int q = 0; q < 8; ++q)
            dst[q] = make_float4(__uint_as_float(v[4 * q]) * inv, __uint_as_float(v[4 * q + 1]) * inv,
                                 __uint_as_float(v[4 * q + 2]) * inv, __uint_as_float(v[4 * q + 3]) * inv);
        }
      }
      if (live && p.n_splits > 1 && c == 0)
        p.part_lse[((int64_t)tok * p.n_splits + split) * H + h] = l > 0.f ? m_ref + __log2f(l) : -INFINITY;
    }
  }

  // ---- tear-down ---------------------------------------------------------------------
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // the peer's last remote arrivals and stores have landed
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

cudaError_t launch_sfa_tc(const SfaParams& p, cudaStream_t s) {
  cudaError_t e = cudaFuncSetAttribute(sfa_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  if (e != cudaSuccess) return e;
  dim3 grid(2 * p.n_splits, p.tv.n_tokens);
  sfa_tc_kernel<<<grid, kThreads, kSmem, s>>>(p);
  return cudaGetLastError();
}

}  // namespace dsa
