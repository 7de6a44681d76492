// Lightning Indexer scoring pass on the 5th-generation tensor cores (tcgen05 + TMA).
//
// Computes, for every query row and every visible key t, the weighted head sum
//   I[t] = sum_h w_h * act(scale_q * scale_k[t] * (q_h . k_t))
// of "Adapting and Optimizing Inference for a New Model Architecture on Ascend",
// section 3.1 (relevance scores against the paged K cache, head weighting), with the
// per-32-element scales of MXFP8 ("Day0 Inference Optimization on Ascend CANN",
// section 3) applied per group.
//
// One persistent CTA per SM walks a contiguous, equal share of the (row, 128-token
// tile) items.  Warp roles:
//   warp 0     TMA producer: two 64-token pages of the K-index cache per tile (each a
//              64 x 128 B box with 128-byte swizzle) into a ring of shared-memory
//              stages (for MXFP8 also the pages' key scales, 256 B each); the row's
//              query [H x d] into one of two query slots;
//   warp 1     one thread issues tcgen05.mma: D[128 tokens x N heads] (f32, TMEM) =
//              K_tile[128 x d] . q[N x d]^T, N = H rounded up to 16; for MXFP8 the
//              block-scaled form applies both sides' group scales in the tensor core;
//   warps 2-9  epilogue, two groups of four warps taking alternate tiles: TMEM lane
//              i = token i; each thread reads its token's head scores with
//              tcgen05.ld, applies scales, activation and head weights, sums over
//              heads, stores one f32 score and counts it in the row's histogram of
//              key top-12-bit bins (what the Top-K pass starts from);
//   warps 10-13  MXFP8 only: one warp per TMEM lane quarter copies each tile's key
//              scales (and, per row, the query's) from shared into tensor memory,
//              where the block-scaled MMA reads them.
// Four TMEM accumulators let the MMA run ahead of both epilogue groups.  Every wait is
// bounded (see sm100::mbar_wait).
#include "sm100.cuh"

namespace dsa {

namespace {

using namespace sm100;

constexpr int kEpiGroups = 2;                    // epilogue groups, alternating tiles
// producer warp, MMA warp, 4 warps per epilogue group; MXFP8 MMAs: 4 scale-factor warps
__host__ __device__ constexpr int tc_threads(int kind, bool fold) {
  return 64 + kEpiGroups * 128 + (kind == 2 && !fold ? 128 : 0);
}
constexpr int kTileTok = 128;
constexpr int kMaxRowsPerLaunch = 1024;
static_assert(kBlockedMaxSeg == kMaxRowsPerLaunch, "a segment of several sequences' rows fits in one launch");

template <int KIND, int D>  // KIND 0: bf16; 1: e4m3 + per-token f32; 2: e4m3 + E8M0 per 32
struct Cfg {
  static constexpr int kElem = KIND == 0 ? 2 : 1;
  static constexpr int kRowBytes = D * kElem;              // bytes of one key / query row
  static constexpr int kRegions = kRowBytes / 128;         // 128-byte swizzle columns per row
  static constexpr int kBoxInner = 128 / kElem;            // elements in one 128-byte piece
  static constexpr int kTileBytes = kTileTok * kRowBytes;  // the keys of a tile
  // MXFP8: the tile's key scales (128 words of four E8M0 bytes) follow its keys
  static constexpr int kStageBytes = kTileBytes + (KIND == 2 ? 1024 : 0);
  // The folded path's epilogue groups wait on the stages themselves: group g takes the
  // tiles n = g mod G and stage n mod S, so with S a multiple of G each group sees every
  // phase of the stages it reads and no parity wait can match a phase two back.
  static constexpr int kStages = KIND == 0 ? 4 : 10;
  static_assert(kStages % kEpiGroups == 0, "stages a multiple of the epilogue groups");
  static constexpr int kRegionStageBytes = kTileTok * 128;  // 16 KB
  static constexpr int kRegionQBytes = 64 * 128;           // 8 KB (up to 64 heads)
  static constexpr int kQSlotBytes = kRegions * kRegionQBytes;
  static constexpr int kKSteps = kRowBytes / 32;           // one MMA consumes 32 bytes of K
  static constexpr int kGroups = KIND == 2 ? D / 32 : 1;   // scale groups per key
  static constexpr int kAccCols = 64;                      // one accumulator: up to 64 heads
  static constexpr int kNumAcc = 4;                        // TMEM accumulator buffers
  // MXFP8: the MMA's scale factors follow the accumulators in tensor memory, 32-column
  // aligned: the keys' for each accumulator in flight, the query's for each query slot
  static constexpr int kSfaCol = kNumAcc * kAccCols;
  static constexpr int kSfbCol = kSfaCol + 32 * kNumAcc;
  static constexpr int kTmemCols = KIND == 2 ? 512 : kNumAcc * kAccCols;
  static_assert(kSfbCol + 64 <= kTmemCols || KIND != 2, "tensor memory budget");
  static constexpr uint32_t kFmt = KIND == 0 ? 1u : 0u;    // bf16 / e4m3
  static constexpr int kSmem = 1024 /*align*/ + kStages * kStageBytes + 2 * kQSlotBytes + 4096 /*bars*/ +
                               4 * (kMaxRowsPerLaunch + 1) * 4 + 4 * kEpiGroups * (64 + 64 * 4 + 4) * 4;
};

struct TcArgs {
  ScoreParams p;
  int32_t row0;   // first query row of this launch
  int32_t nrows;  // rows in this launch
  int32_t seg;    // row-blocked: rows of one sequence in a row of the launch's segments
                  // (nrows is a multiple of it); units are blocks of up to kBlockRows rows
                  // of one segment
};

// Row-blocked unit u of a launch: its first row and its number of rows.
__device__ __forceinline__ void block_unit(const TcArgs& a, int u, int* r0, int* nb) {
  const int per_seg = (a.seg + kBlockRows - 1) / kBlockRows;
  const int sg = u / per_seg, k = u - sg * per_seg;
  *r0 = sg * a.seg + k * kBlockRows;
  *nb = min(kBlockRows, a.seg - k * kBlockRows);
}

// 16 e4m3 values -> f32, exactly.
__device__ __forceinline__ void e4m3x16_to_f32(const uint4& raw, float* out) {
  const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __half2_raw lo = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w[i] & 0xFFFFu), __NV_E4M3);
    const __half2_raw hi = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w[i] >> 16), __NV_E4M3);
    const float2 a = __half22float2(__half2(lo));
    const float2 c = __half22float2(__half2(hi));
    out[4 * i] = a.x;
    out[4 * i + 1] = a.y;
    out[4 * i + 2] = c.x;
    out[4 * i + 3] = c.y;
  }
}

// BLK: row-blocked (bf16 keys, identity activation): the launch's rows come in segments
// of `a.seg` consecutive rows of one sequence (a prefill, or the draft tokens of each
// sequence in multi-token decode); an item is a block of up to kBlockRows rows of one
// segment and one tile of that sequence's keys, read once for the whole block; the MMA's
// N = 64 columns are the block's rows' three split-query terms (p.q: [rows, 3, D]).
// With p.k_scale set (e4m3 keys with per-token scales, dequantised to bf16 beforehand),
// each score is the dot product times its key's scale.
// FOLD: e4m3 keys, identity activation: no tensor cores; the epilogue warps take each
// key's dot product with the folded query q~ (p.qt) straight from the staged tile.
template <int KIND, int D, bool BLK, bool FOLD = false>
__global__ void __launch_bounds__(tc_threads(KIND, FOLD), 1)
    score_tc_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap qmap,
                    const TcArgs a) {
  using C = Cfg<KIND, D>;
  constexpr bool BS = KIND == 2 && !FOLD;  // block-scaled MMAs, scale-factor warps
  constexpr int kThreads = tc_threads(KIND, FOLD);
  const ScoreParams& p = a.p;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  pdl_trigger();  // the next kernel may start its set-up; it waits for this one to finish
  const int H = p.n_heads;
  const int N = (H + 15) / 16 * 16;

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u32 = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024 - (raw_u32 & 1023)) & 1023);
  uint8_t* stages = smem;
  uint8_t* qslots = stages + C::kStages * C::kStageBytes;
  uint64_t* bars = (uint64_t*)(qslots + 2 * C::kQSlotBytes);
  uint64_t* full = bars;
  uint64_t* empty = full + C::kStages;
  uint64_t* acc_full = empty + C::kStages;
  uint64_t* acc_empty = acc_full + C::kNumAcc;
  uint64_t* q_full = acc_empty + C::kNumAcc;
  uint64_t* q_empty = q_full + 2;
  uint64_t* sf_ready = q_empty + 2;  // MXFP8: a tile's scale factors are in TMEM
  uint64_t* drain = sf_ready + C::kStages;
  uint32_t* tmem_base_s = (uint32_t*)(drain + 1);
  volatile int* abort_flag = (volatile int*)(tmem_base_s + 1);
  int* prefix = (int*)(bars + 512);                 // [units + 1] item prefix (unit: a row, or a block)
  int* rowb = prefix + kMaxRowsPerLaunch + 1;       // batch row of each query row
  int* rown = rowb + kMaxRowsPerLaunch + 1;         // visible count of each unit
  int* rn = rown + kMaxRowsPerLaunch + 1;           // visible count of each query row (blocks)
  float* epi = (float*)(rn + kMaxRowsPerLaunch + 1);  // per epilogue warp: w[64], qs[64*4], qtok

  // ---- set-up: barriers, TMEM, per-row metadata and this CTA's item range ----------
  if (tid == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], FOLD ? 4 : 1);  // the MMA's commit, or the four consuming warps
    }
    for (int i = 0; i < C::kNumAcc; ++i) {
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_empty[i], 4);  // the four warps of the group that drains it
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&q_full[i], 1);
      mbar_init(&q_empty[i], 1);
    }
    for (int s = 0; s < C::kStages; ++s) mbar_init(&sf_ready[s], 4);  // the four scale warps
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&kmap);
    tma_prefetch_desc(&qmap);
  }
  if (warp == 1 && !FOLD) {
    tmem_alloc(tmem_base_s, C::kTmemCols);
    tmem_relinquish();
  }
  // visible counts and tiles of every row, then an exclusive scan (one warp)
  const int nunits = BLK ? a.nrows / a.seg * ((a.seg + kBlockRows - 1) / kBlockRows) : a.nrows;
  for (int r = tid; r < a.nrows; r += kThreads) {
    int b, n;
    resolve_token(p.tv, a.row0 + r, &b, &n, p.err);
    rowb[r] = b;
    rn[r] = n;
    if (!BLK) {
      rown[r] = n;
      prefix[r + 1] = (n + kTileTok - 1) / kTileTok;
    }
  }
  if (BLK) {
    __syncthreads();
    for (int u = tid; u < nunits; u += kThreads) {  // a block sees its rows' widest window
      int r0, nb, m = 0;
      block_unit(a, u, &r0, &nb);
      for (int r = r0; r < r0 + nb; ++r) m = max(m, rn[r]);
      rown[u] = m;
      prefix[u + 1] = (m + kTileTok - 1) / kTileTok;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) {
    int carry = 0;
    for (int base = 0; base < nunits; base += 32) {
      const int r = base + lane;
      int v = r < nunits ? prefix[r + 1] : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += u;
      }
      if (r < nunits) prefix[r + 1] = carry + v;
      carry += __shfl_sync(0xffffffffu, v, 31);
    }
    if (lane == 0) prefix[0] = 0;
  }
  __syncthreads();
  const int total = prefix[nunits];
  const int it_begin = (int)((int64_t)total * blockIdx.x / gridDim.x);
  const int it_end = (int)((int64_t)total * (blockIdx.x + 1) / gridDim.x);
  const uint32_t tmem_base = FOLD ? 0u : *tmem_base_s;

  if (warp == 0) {
    // ================================ TMA producer ================================
    // When the query is written by the preceding kernel the producer waits for it (the
    // K-index loads share its in-order issue); a caller-supplied query is read at once.
    if (p.q_dep) pdl_wait();
    // The page ids of the next 32 items are resolved by the warp's lanes at once, one item
    // each (a page-table read costs several hundred cycles: one at a time they would
    // bound the stream); lane 0 then arms and issues the loads in order.
    int stage = 0;
    uint32_t phase = 0;
    uint32_t armed = 0, armed_parity = 0;  // stages with a load issued, and its phase parity
    uint32_t qarmed = 0, qparity = 0;      // the same for the two query slots
    int r = 0, cur_row = -1, qcount = 0;
    bool stop = false;
    // (streamed keys leave L2 first: the scores and histograms written meanwhile stay
    // there for the selection pass)
    const uint64_t l2_evict_first = l2_policy_evict_first();
    for (int it0 = it_begin; it0 < it_end && !stop; it0 += 32) {
      const int mine = it0 + lane;
      int lr = r, lpg0 = -1, lpg1 = -1;
      if (mine < it_end) {
        while (prefix[lr + 1] <= mine) ++lr;
        const int tile = mine - prefix[lr];
        int br = lr;
        if (BLK) {
          int unb;
          block_unit(a, lr, &br, &unb);
        }
        const int npages = (rown[lr] + kPage - 1) / kPage;
        if (2 * tile < npages) lpg0 = physical_page(p.tv, rowb[br], 2 * tile, p.err);
        if (2 * tile + 1 < npages) lpg1 = physical_page(p.tv, rowb[br], 2 * tile + 1, p.err);
      }
      const int nb = min(32, it_end - it0);
      for (int k = 0; k < nb; ++k) {
        const int pg[2] = {__shfl_sync(0xffffffffu, lpg0, k), __shfl_sync(0xffffffffu, lpg1, k)};
        int ok = 1;
        if (lane == 0) {
          const int it = it0 + k;
          while (prefix[r + 1] <= it) ++r;
          if (!FOLD && r != cur_row) {
            cur_row = r;
            int ur0 = r, unb = 1;
            if (BLK) block_unit(a, r, &ur0, &unb);
            const int slot = qcount & 1;
            ok = mbar_wait(&q_empty[slot], ((qcount >> 1) & 1) ^ 1, abort_flag, p.err, p.wait_limit);
            if (ok) {
              mbar_arrive_expect_tx(&q_full[slot], C::kRegions * H * 128);
              qarmed |= 1u << slot;
              qparity = (qparity & ~(1u << slot)) | ((uint32_t)((qcount >> 1) & 1) << slot);
              const uint32_t qdst = smem_u32(qslots + slot * C::kQSlotBytes);
              for (int g = 0; g < C::kRegions; ++g)
                tma_load_2d(qdst + g * C::kRegionQBytes, &qmap, &q_full[slot], g * C::kBoxInner,
                            BLK ? 3 * (a.row0 + ur0) : (a.row0 + r) * H);
              ++qcount;
            }
          }
          if (ok) ok = mbar_wait(&empty[stage], phase ^ 1, abort_flag, p.err, p.wait_limit);
          if (ok) {
            uint32_t bytes = 0;
            for (int u = 0; u < 2; ++u)
              if (pg[u] >= 0) bytes += kPage * C::kRowBytes + (BS ? kPage * 4 : 0);
            mbar_arrive_expect_tx(&full[stage], bytes);
            armed |= 1u << stage;
            armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
            const uint32_t sdst = smem_u32(stages + stage * C::kStageBytes);
            for (int u = 0; u < 2; ++u) {
              if (pg[u] < 0) continue;
              for (int g = 0; g < C::kRegions; ++g)  // keys are read once: evict them first
                tma_load_2d_hint(sdst + g * C::kRegionStageBytes + u * (kPage * 128), &kmap, &full[stage],
                                 g * C::kBoxInner, pg[u] * kPage, l2_evict_first);
              if (BS)  // the page's 64 key scale words (a 16-byte aligned 256-byte run)
                bulk_load(sdst + C::kTileBytes + u * (kPage * 4), (const uint8_t*)p.k_scale + (int64_t)pg[u] * kPage * 4,
                          kPage * 4, &full[stage]);
            }
            if (++stage == C::kStages) {
              stage = 0;
              phase ^= 1;
            }
          }
        }
        if (!__shfl_sync(0xffffffffu, ok, 0)) {
          stop = true;
          break;
        }
      }
      r = __shfl_sync(0xffffffffu, r, 0);
    }
    if (lane == 0 && *abort_flag) {
      // let every copy still in flight (key tiles and queries) land before the shared
      // memory is released
      for (int st = 0; st < C::kStages; ++st) {
        if (!(armed >> st & 1)) continue;
        const long long t0 = clock64();
        while (!mbar_try_wait(smem_u32(&full[st]), (armed_parity >> st) & 1) && clock64() - t0 < kWaitLimitCycles) {
        }
      }
      for (int sl = 0; sl < 2; ++sl) {
        if (!(qarmed >> sl & 1)) continue;
        const long long t0 = clock64();
        while (!mbar_try_wait(smem_u32(&q_full[sl]), (qparity >> sl) & 1) && clock64() - t0 < kWaitLimitCycles) {
        }
      }
    }
  } else if (warp == 1) {
    // ================================ MMA issuer ==================================
    if (lane == 0 && !FOLD) {
      const uint32_t idesc_v = idesc(128, N, C::kFmt, C::kFmt);
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;  // acc cycles through kNumAcc buffers
      int r = 0, cur_row = -1, qcount = 0, slot = 0;
      for (int it = it_begin; it < it_end; ++it) {
        while (prefix[r + 1] <= it) ++r;
        if (r != cur_row) {
          cur_row = r;
          slot = qcount & 1;
          if (!mbar_wait(&q_full[slot], (qcount >> 1) & 1, abort_flag, p.err, p.wait_limit)) break;
          ++qcount;
        }
        if (!mbar_wait(&full[stage], phase, abort_flag, p.err, p.wait_limit)) break;
        if (BS && !mbar_wait(&sf_ready[stage], phase, abort_flag, p.err, p.wait_limit)) break;
        if (!mbar_wait(&acc_empty[acc], acc_phase ^ 1, abort_flag, p.err, p.wait_limit)) break;
        tc_fence_after();
        const uint32_t a0 = smem_u32(stages + stage * C::kStageBytes);
        const uint32_t b0 = smem_u32(qslots + slot * C::kQSlotBytes);
        const uint32_t d0 = tmem_base + acc * C::kAccCols;
#pragma unroll
        for (int k = 0; k < C::kKSteps; ++k) {
          const int g = k / 4, off = (k % 4) * 32;
          const uint64_t ad = desc_sw128(a0 + g * C::kRegionStageBytes + off);
          const uint64_t bd = desc_sw128(b0 + g * C::kRegionQBytes + off);
          if (KIND == 0) {
            mma_f16(d0, ad, bd, idesc_v, k > 0);
          } else if (KIND == 1) {
            mma_f8(d0, ad, bd, idesc_v, k > 0);
          } else {  // K block k: byte k of each scale word
            mma_mxf8(d0, ad, bd, idesc_mx(128, N, k, k), tmem_base + C::kSfaCol + 32 * acc,
                     tmem_base + C::kSfbCol + 32 * slot, k > 0);
          }
        }
        tc_commit(&empty[stage]);
        tc_commit(&acc_full[acc]);
        if (it + 1 == it_end || prefix[r + 1] == it + 1) tc_commit(&q_empty[slot]);
        if (++stage == C::kStages) {
          stage = 0;
          phase ^= 1;
        }
        if (++acc == C::kNumAcc) {
          acc = 0;
          acc_phase ^= 1;
        }
      }
      // every MMA issued above has completed once `drain` flips
      tc_commit(drain);
      const long long t0 = clock64();
      while (!mbar_try_wait(smem_u32(drain), 0) && clock64() - t0 < kWaitLimitCycles) {
      }
    }
  } else if (BS && warp >= 2 + 4 * kEpiGroups) {
    // ============================ scale factors (MXFP8) ===========================
    // Each lane quarter of the tensor core reads the scale factors from its own 32
    // TMEM lanes, so each of the four warps writes the same words into its quarter:
    // row j of the MMA (key j of the tile, head j of the query) at lane j % 32, column
    // j / 32, one byte per 32-element group.  A tile's key scales go to the columns of
    // its accumulator once that accumulator is free (its previous MMAs are done); the
    // query's go to its slot's columns with the row's first tile, which the producer
    // loads only after the slot's previous row has finished.
    const uint32_t lq = tmem_base + ((uint32_t)((warp & 3) * 32) << 16);
    int stage = 0, acc = 0, r = 0, cur_row = -1, qcount = 0;
    uint32_t phase = 0, acc_phase = 0;
    for (int it = it_begin; it < it_end; ++it) {
      while (prefix[r + 1] <= it) ++r;
      bool ok = true;
      if (lane == 0) {
        ok = mbar_wait(&full[stage], phase, abort_flag, p.err, p.wait_limit) &&
             mbar_wait(&acc_empty[acc], acc_phase ^ 1, abort_flag, p.err, p.wait_limit);
      }
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      __syncwarp();
      tc_fence_after();
      if (r != cur_row) {
        cur_row = r;
        const int slot = qcount++ & 1;
        const int64_t qrow = (int64_t)(a.row0 + r) * H;
        const uint32_t* qs = (const uint32_t*)p.q_scale;
        tmem_st2(lq + C::kSfbCol + 32 * slot, lane < H ? qs[qrow + lane] : 0x7F7F7F7Fu,
                 32 + lane < H ? qs[qrow + 32 + lane] : 0x7F7F7F7Fu);
      }
      const uint32_t* ks = (const uint32_t*)(stages + stage * C::kStageBytes + C::kTileBytes);
      tmem_st4(lq + C::kSfaCol + 32 * acc, ks[lane], ks[32 + lane], ks[64 + lane], ks[96 + lane]);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sf_ready[stage]);
      if (++stage == C::kStages) {
        stage = 0;
        phase ^= 1;
      }
      if (++acc == C::kNumAcc) {
        acc = 0;
        acc_phase ^= 1;
      }
    }
  } else {
    // ================================ epilogue ====================================
    // Group g drains the tiles n with n % kEpiGroups == g; tile n sits in accumulator
    // n % kNumAcc.  Within a group, TMEM lane i (warp quarter q = warp & 3) = token i.
    // The scores and histograms it writes share workspace with the previous pass, so
    // it first waits for the previous kernel (the loads and MMAs above need not).
    pdl_wait();
    const int grp = (warp - 2) / 4;
    const int quarter = warp & 3;
    const int i = quarter * 32 + lane;
    if constexpr (BLK) {
      // token i of the tile against every row of the block: column 3 j + e is term e of
      // row j, the row's score their sum; each row masks its own causal window
      int r = 0;
      for (int it = it_begin; it < it_end; ++it) {
        while (prefix[r + 1] <= it) ++r;
        const int n = it - it_begin;
        if (n % kEpiGroups != grp) continue;
        const int acc = n % C::kNumAcc;
        const uint32_t acc_phase = (uint32_t)(n / C::kNumAcc) & 1u;
        const int t = (it - prefix[r]) * kTileTok + i;
        int r0, nb;
        block_unit(a, r, &r0, &nb);
        const int pg = t < rown[r] ? physical_page(p.tv, rowb[r0], t >> 6, nullptr) : -1;
        const float ksc = (p.k_scale && pg >= 0) ? ((const float*)p.k_scale)[(int64_t)pg * kPage + (t & 63)] : 1.f;
        bool ok = true;
        if (lane == 0) ok = mbar_wait(&acc_full[acc], acc_phase, abort_flag, p.err, p.wait_limit);
        if (!__shfl_sync(0xffffffffu, ok, 0)) break;
        __syncwarp();
        tc_fence_after();
        const uint32_t tbase = tmem_base + ((uint32_t)(quarter * 32) << 16) + acc * C::kAccCols;
        uint32_t v0[32], v1[32];
        tmem_ld32(tbase, v0);
        tmem_ld32(tbase + 32, v1);
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acc_empty[acc]);
#pragma unroll
        for (int j = 0; j < kBlockRows; ++j) {
          if (j < nb && t < rn[r0 + j]) {
            const float c0 = __uint_as_float(3 * j < 32 ? v0[(3 * j) & 31] : v1[(3 * j) & 31]);
            const float c1 = __uint_as_float(3 * j + 1 < 32 ? v0[(3 * j + 1) & 31] : v1[(3 * j + 1) & 31]);
            const float c2 = __uint_as_float(3 * j + 2 < 32 ? v0[(3 * j + 2) & 31] : v1[(3 * j + 2) & 31]);
            const float v = pg >= 0 ? ((c0 + c1) + c2) * ksc : -INFINITY;
            const int64_t grow = a.row0 + r0 + j;
            p.scores[grow * p.score_stride + t] = v;
            atomicAdd(p.hist + grow * kTopkBins + (score_key(v) >> 20), 1u);
          }
        }
      }
    } else if constexpr (FOLD) {
      // token i of the tile: its key (one 128-byte swizzled row of e4m3) against q~, the
      // key's scale per token or per 32-element group applied to the partial sums
      static_assert(KIND != 0 && D == 128, "folded scoring: e4m3 keys of 128 elements");
      float* qt_s = epi + (warp - 2) * (64 + 64 * 4 + 4);  // this warp's copy of q~
      int r = 0, cur_row = -1;
      for (int it = it_begin; it < it_end; ++it) {
        while (prefix[r + 1] <= it) ++r;
        const int n = it - it_begin;
        if (n % kEpiGroups != grp) continue;
        const int grow = a.row0 + r;
        if (r != cur_row) {
          cur_row = r;
          __syncwarp();
          for (int d = lane; d < D; d += 32) qt_s[d] = p.qt[(int64_t)grow * D + d];
          __syncwarp();
        }
        const int stage = n % C::kStages;
        const uint32_t par = (uint32_t)(n / C::kStages) & 1u;
        const int t = (it - prefix[r]) * kTileTok + i;
        const bool valid = t < rown[r];
        const int pg = valid ? physical_page(p.tv, rowb[r], t >> 6, nullptr) : -1;
        float ks[4] = {1.f, 1.f, 1.f, 1.f};
        if (pg >= 0) {
          const int64_t krow = (int64_t)pg * kPage + (t & 63);
          if (KIND == 1) {
            ks[0] = ((const float*)p.k_scale)[krow];
          } else {
            const uint32_t k4 = *(const uint32_t*)((const uint8_t*)p.k_scale + krow * 4);
#pragma unroll
            for (int g = 0; g < 4; ++g) ks[g] = e8m0_to_f32((k4 >> (8 * g)) & 0xFF);
          }
        }
        bool ok = true;
        if (lane == 0) ok = mbar_wait(&full[stage], par, abort_flag, p.err, p.wait_limit);
        if (!__shfl_sync(0xffffffffu, ok, 0)) break;
        __syncwarp();
        const uint8_t* krow_s = stages + stage * C::kStageBytes + i * 128;
        float acc = 0.f;
#pragma unroll
        for (int g = 0; g < 4; ++g) {  // 32-element groups, two 16-byte chunks each
          float ag = 0.f;
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            const int u = 2 * g + hh;
            float f[16];
            e4m3x16_to_f32(*(const uint4*)(krow_s + ((u ^ (i & 7)) << 4)), f);
            const float4* q4 = (const float4*)(qt_s + 16 * u);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float4 qq = q4[e];
              ag = fmaf(f[4 * e], qq.x, ag);
              ag = fmaf(f[4 * e + 1], qq.y, ag);
              ag = fmaf(f[4 * e + 2], qq.z, ag);
              ag = fmaf(f[4 * e + 3], qq.w, ag);
            }
          }
          acc += KIND == 2 ? ag * ks[g] : ag;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[stage]);  // this warp has read its 32 keys
        if (valid) {
          const float v = pg >= 0 ? (KIND == 1 ? acc * ks[0] : acc) : -INFINITY;
          p.scores[(int64_t)grow * p.score_stride + t] = v;
          atomicAdd(p.hist + (int64_t)grow * kTopkBins + (score_key(v) >> 20), 1u);
        }
      }
    } else {
    // (MXFP8 accumulators arrive with both sides' scales applied by the MMA)
    float* w_s = epi + (warp - 2) * (64 + 64 * 4 + 4);
    int r = 0, cur_row = -1;
    float qtok = 1.f;
    for (int it = it_begin; it < it_end; ++it) {
      while (prefix[r + 1] <= it) ++r;
      const int n = it - it_begin;
      if (n % kEpiGroups != grp) continue;
      const int acc = n % C::kNumAcc;
      const uint32_t acc_phase = (uint32_t)(n / C::kNumAcc) & 1u;
      const int grow = a.row0 + r;
      if (r != cur_row) {
        cur_row = r;
        __syncwarp();
        for (int h = lane; h < H; h += 32) w_s[h] = p.head_w[(int64_t)grow * H + h];
        qtok = (KIND == 1) ? ((const float*)p.q_scale)[grow] : 1.f;
        __syncwarp();
      }
      const int tile = it - prefix[r];
      const int t = tile * kTileTok + i;
      const bool valid = t < rown[r];
      int pg = -1;
      if (valid) pg = physical_page(p.tv, rowb[r], t >> 6, nullptr);
      const float ks = (KIND == 1 && pg >= 0) ? ((const float*)p.k_scale)[(int64_t)pg * kPage + (t & 63)] : 1.f;
      bool ok = true;
      if (lane == 0) ok = mbar_wait(&acc_full[acc], acc_phase, abort_flag, p.err, p.wait_limit);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      __syncwarp();
      tc_fence_after();
      const uint32_t tbase = tmem_base + ((uint32_t)(quarter * 32) << 16) + acc * C::kAccCols;
      float part[4] = {0.f, 0.f, 0.f, 0.f};  // four independent sums over heads
      {
        uint32_t v0[32], v1[32];
        tmem_ld32(tbase, v0);
        if (H > 32) tmem_ld32(tbase + 32, v1);
        tmem_ld_wait();
        const float sc = (KIND == 1) ? qtok * ks : 1.f;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          if (j < H) {
            float x = __uint_as_float(v0[j]);
            if (KIND == 1) x *= sc;
            if (p.act == DSA_ACT_RELU) x = fmaxf(x, 0.f);
            part[j & 3] += x * w_s[j];
          }
        }
        if (H > 32) {
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            if (32 + j < H) {
              float x = __uint_as_float(v1[j]);
              if (KIND == 1) x *= sc;
              if (p.act == DSA_ACT_RELU) x = fmaxf(x, 0.f);
              part[j & 3] += x * w_s[32 + j];
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[acc]);
      if (valid) {
        const float v = pg >= 0 ? (part[0] + part[1]) + (part[2] + part[3]) : -INFINITY;
        p.scores[(int64_t)grow * p.score_stride + t] = v;
        atomicAdd(p.hist + (int64_t)grow * kTopkBins + (score_key(v) >> 20), 1u);
      }
    }
    }  // per-row epilogue
  }

  // ---- tear-down ---------------------------------------------------------------------
  tc_fence_before();
  __syncthreads();
  if (warp == 1 && !FOLD) {
    tc_fence_after();
    tmem_dealloc(tmem_base, C::kTmemCols);
  }
}

// ---- host side: launch ---------------------------------------------------------------
template <int KIND, int D, bool BLK = false, bool FOLD = false>
cudaError_t launch_tc(const ScoreParams& p, cudaStream_t s) {
  using C = Cfg<KIND, D>;
  static_assert(C::kSmem <= 232448, "shared memory budget");
  CUtensorMap kmap, qmap;
  if (!make_tma_2d_sw128(&kmap, p.k, (uint64_t)p.tv.num_pages * kPage, C::kElem, D, kPage)) return cudaErrorInvalidValue;
  static std::atomic<int> smem_set[kMaxDevices];
  cudaError_t e = set_smem_once(score_tc_kernel<KIND, D, BLK, FOLD>, C::kSmem, smem_set);
  if (e != cudaSuccess) return e;
  const int sms = device_sm_count();
  // the query: [tokens * heads, D], boxes of one token's heads; blocked: [tokens * 3, D],
  // boxes of 64 rows (a block's 21 tokens x 3 terms, and one spare row)
  if (!make_tma_2d_sw128(&qmap, p.q, (uint64_t)p.tv.n_tokens * (BLK ? 3 : p.n_heads), C::kElem, D,
                         BLK ? 64 : p.n_heads))
    return cudaErrorInvalidValue;
  // row-blocked: launches start at segment boundaries (a segment longer than a launch
  // is one sequence, cut anywhere)
  const int seg = BLK ? p.seg_rows : 1;
  const int per_launch = seg >= kMaxRowsPerLaunch ? kMaxRowsPerLaunch : kMaxRowsPerLaunch / seg * seg;
  for (int row0 = 0; row0 < p.tv.n_tokens; row0 += per_launch) {
    TcArgs a;
    a.p = p;
    a.row0 = row0;
    a.nrows = p.tv.n_tokens - row0 < per_launch ? p.tv.n_tokens - row0 : per_launch;
    a.seg = seg < a.nrows ? seg : a.nrows;
    e = launch_pdl(score_tc_kernel<KIND, D, BLK, FOLD>, dim3(sms), dim3(tc_threads(KIND, FOLD)), C::kSmem, s, kmap, qmap, a);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace

long long sm100_default_wait_limit() { return kWaitLimitCycles; }

bool score_tc_supported(dsa_dtype_t dt, int dim, int n_heads) {
  if (n_heads < 1 || n_heads > 64) return false;
  if (dt == DSA_BF16) return dim == 64 || dim == 128;
  return dim == 128;
}

bool score_fold_supported(dsa_dtype_t dt, dsa_scale_t sk, dsa_act_t act, int dim) {
  // (MX keys measured slower this way than through the per-head tensor-core kernel)
  return dt == DSA_E4M3 && sk == DSA_SCALE_PER_TOKEN_F32 && act == DSA_ACT_IDENTITY && dim == 128;
}

cudaError_t launch_score_fold(const ScoreParams& p, dsa_scale_t sk, const float* qt, cudaStream_t s) {
  ScoreParams f = p;
  f.qt = qt;
  return sk == DSA_SCALE_PER_TOKEN_F32 ? launch_tc<1, 128, false, true>(f, s) : launch_tc<2, 128, false, true>(f, s);
}

cudaError_t launch_score_tc_blocked(const ScoreParams& p, cudaStream_t s) {
  ScoreParams b = p;
  b.n_heads = 64;  // N: 21 rows x 3 terms + 1
  return p.dim == 64 ? launch_tc<0, 64, true>(b, s) : launch_tc<0, 128, true>(b, s);
}

cudaError_t launch_score_tc(const ScoreParams& p, dsa_dtype_t dt, dsa_scale_t sk, cudaStream_t s) {
  if (dt == DSA_BF16) return p.dim == 64 ? launch_tc<0, 64>(p, s) : launch_tc<0, 128>(p, s);
  if (sk == DSA_SCALE_PER_TOKEN_F32) return launch_tc<1, 128>(p, s);
  return launch_tc<2, 128>(p, s);
}

}  // namespace dsa
