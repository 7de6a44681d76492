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
//     over its 288 "own" dims: latent [256c, 256c + 256) and rope [512 + 32c, +32).
//     Each CTA gathers its 512 latent bytes and its 64 rope bytes of every selected
//     row (the pair reads each 1152-byte row once from DRAM).
//   * Each CTA computes partial logits S_c = Q[:, own] . KV[:, own]^T (tcgen05, A = Q
//     from tensor memory, B = gathered rows in shared memory), multiplies them by
//     softmax_scale * log2(e), rounds them to fp16 (relative 2^-11, below the bf16
//     rounding P gets anyway), sends them to its peer through distributed shared
//     memory (each warp stages its 32 rows and moves them with one bulk copy, counted
//     in bytes on the peer's mbarrier) and adds the peer's part: both CTAs hold the
//     same S = S_0 + S_1 of the same rounded halves.
//   * Online softmax per head row (thread = row, no shuffles), base 2; the reference
//     maximum only moves when a tile's maximum exceeds it by 8 (2^8 headroom), and O is
//     then rescaled in tensor memory.
//   * P (bf16) goes to shared memory; O[128 x 256] += P . V with V read MN-major from
//     the same shared-memory rows the logits used.
// Warp roles (sixteen warps): warps 0-2 gather rows with TMA gather4 into a 4-stage ring
// of swizzled rows, each lane issuing its own gathers (a gather's cost is in its issue);
// warp 3 (converged, one elected lane) issues each MMA as soon as its inputs are ready;
// warps 4-7 (senders) load each tile's partial logits, round them and send them to the
// peer; warps 8-11 and 12-15 (finishers) take key columns 0-31 and 32-63 of each tile:
// each rounds its own half of the logits as the senders do, adds the peer's part, meets
// its partner warp (same 32 head rows) to share the row maxima, runs its half of the
// softmax and stores its half of P; warps 8-11 then run the epilogue.  Sending tile
// n + 1 and finishing tile n thus run at the same time.  Tensor memory (512 columns): O [0,256), two logit buffers
// S0 [256,320) and S1 [320,384), Q latent [384,512).  Tile n uses logit buffer n & 1;
// its P (bf16) is written over the peer's partial logits of tile n in the receive
// buffer n & 1 (same 128-byte-swizzled rows, each thread its own row), and P.V(n)'s
// completion hands that buffer back to the peer.  So QK(n + 1), the softmax of tile n
// and P.V(n - 1) proceed at the same time; QK(n) only waits for the senders to have
// read S(n - 2).  Q's rope dims are an MMA operand in shared memory.  Every wait is
// bounded.  Shared memory per stage: 4 latent regions of 64 rows x 128 B (128-byte
// swizzle) + 1 rope region of 64 rows x 64 B (64-byte swizzle).
#include <cuda_fp16.h>

#include "sm100.cuh"

namespace dsa {

namespace {

using namespace sm100;

constexpr int kGatherWarps = 3;                  // warps 0-2 gather (TMA), warp 3 issues MMAs
constexpr int kMmaWarp = kGatherWarps;
constexpr int kSendWarp0 = kMmaWarp + 1;          // warps 4-7 load and send the partial logits
constexpr int kFinWarp0 = kSendWarp0 + 4;         // warps 8-11 finish key columns 0-31 of each tile and run
                                                  // the epilogue
constexpr int kFinWarpB0 = kFinWarp0 + 4;         // warps 12-15 finish key columns 32-63
constexpr int kExtraWarp0 = kFinWarpB0 + 4;       // warps 16-19: gather too (bf16 cache) or convert
                                                  // the gathered FP8 rows (FP8 cache)
constexpr int kThreads = (kExtraWarp0 + 4) * 32;
constexpr int kTok = 64;                         // selected positions per tile
constexpr int kStages = 4;
constexpr int kRegion = kTok * 128;              // 64 rows x 128 B
constexpr int kRopeRegion = kTok * 64;           // 64 rows x 64 B
constexpr int kGathers = (kTok / 4) * 5;         // per tile: 16 groups of 4 slots x 5 pieces
constexpr int kStageBytes = 4 * kRegion + kRopeRegion;  // 4 latent regions + 1 rope region
constexpr int kXchBytes = 128 * kTok * 2;        // one fp16 partial-logit tile (128 rows x 128 B)
constexpr int kMaxSplitLen = kMaxTopK;
constexpr uint32_t kColO = 0, kColS = 256, kColQl = 384;  // S buffer b: kColS + 64 b
constexpr int kQRegion = 128 * 128;                // Q latent staging: 4 regions of 128 rows x 128 B
static_assert(4 * kQRegion <= 2 * kStageBytes, "Q latent staging fits in stage buffers 2-3");
constexpr int kQropeBytes = 128 * 64;             // Q rope (own 32 dims) [128 rows][64 B], 64-byte swizzle
constexpr int kMaxXBytes = 2 * 2 * 128 * 4;       // finisher pairs' row maxima [tile parity][half][row]
constexpr int kSmem = 1024 + kStages * kStageBytes + kQropeBytes + 3 * kXchBytes + kMaxXBytes + kMaxSplitLen * 4 + 512;
static_assert(kSmem <= 232448, "shared memory budget");
// FP8 latent cache: per tile and group of 4 slots, two 128-byte pieces of e4m3 codes
// (this CTA's 256 latent dims) and the 64-byte rope piece; plus one 16-byte copy of each
// row's four tile scales into a per-stage scale area [64 rows][4] f32, on the load/store
// path (cp.async), beside the 48 gathers of a tile; the 48 copying lanes arrive on
// kv_full as their copies land.
constexpr int kGathersFp8 = (kTok / 4) * 3;
constexpr int kScaleLanes = kGatherWarps * 32 - kGathersFp8;  // lanes of warps 0-2 past the gathers
constexpr int kConvWarps = 4;                                 // warps 16-19
constexpr int kScaleArea = kTok * 16;
constexpr int kSmemFp8 = kSmem + kStages * kScaleArea;
static_assert(kSmemFp8 <= 232448, "shared memory budget (FP8 latent)");
static_assert(kScaleLanes == 48 && kTok - kScaleLanes <= kScaleLanes, "scale rows j and j + 48 cover the tile");
// Sibling merge (two splits in one cluster): outbox and inbox of 128 rows x 128 f32
// columns plus 128 (m, l) pairs each, in the stage buffers.
constexpr uint32_t kSibBytes = 128 * 256 + 128 * 8;  // 128 rows x 128 fp16 columns, then (m, l) per row
static_assert(2 * kSibBytes <= kStages * kStageBytes, "sibling merge buffers fit in the stage buffers");

// Packed bf16 product (round to nearest even; subnormal inputs and results kept).
__device__ __forceinline__ uint32_t mul_bf16x2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.bf16x2 %0, %1, %2;\n" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// 16 e4m3 codes times a scale -> 16 bf16, as 8 packed pairs, without the conversion pipe
// (which the softmax warps keep busy): each code's bits s.eeee.mmm are spread into a
// bf16 field as s.0000eeee.mmm0000, which encodes exactly code * 2^-120 (e = 0, the
// E4M3 subnormals, becoming bf16 subnormals), then two packed products: by 2^60 (exact)
// and by sc60 = bf16(scale * 2^60), one rounding.  (The scale enters rounded to bf16:
// exact for power-of-two scales, else within 2^-9 relative of the f32 scale.)
__device__ __forceinline__ void e4m3x16_scaled_to_bf16(const uint4& raw, uint32_t sc60, uint32_t (&out)[8]) {
  const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
  constexpr uint32_t kTwo60 = 0x5D805D80u;  // bf16 pair (2^60, 2^60)
#pragma unroll
  for (int i = 0; i < 4; ++i) {
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
      const uint32_t t = __byte_perm(w[i], 0u, hf ? 0x4342u : 0x4140u);  // bytes 2hf, 2hf+1 in 16-bit lanes
      const uint32_t f = ((t << 4) & 0x07F007F0u) | ((t << 8) & 0x80008000u);
      out[2 * i + hf] = mul_bf16x2(mul_bf16x2(f, kTwo60), sc60);
    }
  }
}

// Launched in clusters of two CTAs (the pair), or four (two splits x the pair) when the
// two splits of a token merge inside the cluster.
// FP8: the latent cache holds e4m3 codes with an f32 scale per 128-dim tile and bf16
// rope dims.  The codes of this CTA's 256 latent dims land (TMA gather4, 128-byte
// swizzled rows) in latent regions 2 and 3 of the stage, the row scales in the stage's
// scale area and the rope dims in the rope region as for a bf16 cache; then the gather
// warps turn each row into bf16 (code x scale, rounded to nearest even: exact when the
// scale is a power of two) in latent regions 0-3, the layout the MMAs read.  Each row's
// four 64-dim output pieces are written by four lanes of one warp after all four have
// read their codes (the codes of row r sit in row r of regions 2-3, which pieces 2-3 of
// row r overwrite), and kv_conv[stage] tells the MMA issuer that the tile is ready.
template <bool FP8>
__global__ void __launch_bounds__(kThreads, 1)
    sfa_tc_kernel(const __grid_constant__ CUtensorMap kvmap, const __grid_constant__ CUtensorMap ropemap,
                  const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap qropemap, SfaParams p) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = cluster_rank();  // 2 * (split within the cluster) + c
  const uint32_t c = rank & 1u;
  const uint32_t peer = rank ^ 1u;
  const int split = blockIdx.x >> 1, tok = blockIdx.y;
  const int H = p.n_heads;
  pdl_trigger();  // the next kernel may start its set-up; it waits for this one to finish

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u32 = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024 - (raw_u32 & 1023)) & 1023);
  uint8_t* stages = smem;
  uint8_t* qrope = stages + kStages * kStageBytes;            // Q rope operand
  uint8_t* xch = qrope + kQropeBytes;                         // [2][128 rows][64 fp16] peer partials, then P
  uint8_t* stg = xch + 2 * kXchBytes;                         // [128 rows][64 fp16] own partial, outbound
  float* maxx = (float*)(stg + kXchBytes);                    // [2][2][128] finisher pairs' row maxima
  int32_t* rowid = (int32_t*)((uint8_t*)maxx + kMaxXBytes);   // cache row of each slot or -1
  uint64_t* bars = (uint64_t*)(rowid + kMaxSplitLen);
  uint64_t* kv_full = bars;
  uint64_t* kv_empty = kv_full + kStages;
  uint64_t* q_ready = kv_empty + kStages;
  uint64_t* s_full = q_ready + 1;     // [2] per logit buffer: QK done
  uint64_t* s_free = s_full + 2;      // [2]: every softmax warp has read the logits
  uint64_t* p_full = s_free + 2;      // [2] per receive buffer: P stored
  uint64_t* pv_done = p_full + 2;     // [2]: P.V done (P read, O updated)
  uint64_t* xch_full = pv_done + 2;   // [2]: peer partial of tile t in buffer t & 1
  uint64_t* xch_empty = xch_full + 2;  // [2]: the peer is done with our partial of tile t (its P.V ran)
  uint64_t* drain = xch_empty + 2;
  uint64_t* q_tma = drain + 1;    // Q (own dims) landed in shared memory
  uint64_t* m_ready = q_tma + 1;  // sibling merge: the sibling's inbox is free
  uint64_t* m_full = m_ready + 1; // sibling merge: the sibling's columns arrived
  uint64_t* kv_conv = m_full + 1;  // [kStages] (FP8): the tile's rows are bf16 in the stage
  uint32_t* tmem_base_s = (uint32_t*)(kv_conv + kStages);
  volatile int* abort_flag = (volatile int*)(tmem_base_s + 1);
  int* last_valid_s = (int*)(abort_flag + 1);                // last slot holding a selected row
  float* scale_area = (float*)(bars + 64);                   // (FP8) [kStages][64 rows][4] f32

  int b, n_vis;
  resolve_token(p.tv, tok, &b, &n_vis, nullptr);
  const int j_begin = split * p.split_len;
  const int j_end = min(p.top_k, j_begin + p.split_len);
  const int ntok = max(0, j_end - j_begin);
  const int n_tiles = (ntok + kTok - 1) / kTok;

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&kv_full[s], FP8 ? kGatherWarps + kScaleLanes : kGatherWarps + 4);
      mbar_init(&kv_empty[s], 1);
    }
    mbar_init(q_ready, 4);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&s_free[i], 12);  // the four senders and the eight finishers have read the logits
      mbar_init(&p_full[i], 8);   // both halves of every row of P stored
      mbar_init(&pv_done[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&xch_full[i], 1);   // armed locally per tile; the peer's four copies count bytes
      mbar_init(&xch_empty[i], 1);  // the peer's P.V(t) completion, multicast by its MMA thread
    }
    mbar_init(drain, 1);
    mbar_init(q_tma, 1);
    mbar_init(m_ready, 1);
    mbar_init(m_full, 1);
    for (int i = 0; i < kStages; ++i) mbar_init(&kv_conv[i], kConvWarps);
    *abort_flag = 0;
    *last_valid_s = -1;
    // the peer's partial logits of tiles 0 and 1 may arrive as soon as the cluster syncs
    for (int t = 0; t < 2 && t < n_tiles; ++t) mbar_arrive_expect_tx(&xch_full[t], kXchBytes);
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(tmem_base_s, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_base_s;
  // Q does not depend on the previous kernel: fetch it while that one finishes.  Its
  // latent own dims land (TMA, 128-byte swizzle) in stage buffers 2-3, idle until tile
  // 2's gathers; its rope own dims land directly as the 64-byte-swizzled MMA operand.
  uint8_t* qstage = stages + 2 * kStageBytes;
  if (warp == kMmaWarp && lane == 0) {
    mbar_arrive_expect_tx(q_tma, (uint32_t)H * (4 * 128 + 64));
#pragma unroll
    for (int q = 0; q < 4; ++q)
      tma_load_2d(smem_u32(qstage + q * kQRegion), &qmap, q_tma, 256 * (int)c + 64 * q, tok * H);
    tma_load_2d(smem_u32(qrope), &qropemap, q_tma, 512 + 32 * (int)c, tok * H);
    tma_prefetch_desc(&kvmap);
    tma_prefetch_desc(&ropemap);
  }
  __syncwarp();
  cluster_arrive();  // this CTA's barriers exist (the wait comes before any remote traffic)
  if (warp >= kSendWarp0 && warp < kFinWarp0) {
    // each sending thread moves its head row h of the latent part into tensor memory
    // (packed bf16 pairs); rows past the head count are zero, in the rope operand too.
    // Q is an input: this runs before the dependency wait, off the gathers' path
    const int quarter = warp & 3;
    const int h = quarter * 32 + lane;  // head row == TMEM lane
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const bool live = h < H;
    bool good = true;
    if (lane == 0) good = mbar_wait(q_tma, 0, abort_flag, p.err);
    good = __shfl_sync(0xffffffffu, good, 0);
#pragma unroll 1
    for (int q = 0; q < 4; ++q) {
      uint32_t w[32];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const uint4 x = (live && good) ? *(const uint4*)(qstage + q * kQRegion + h * 128 + ((u ^ (h & 7)) << 4))
                                       : make_uint4(0, 0, 0, 0);
        w[4 * u] = x.x;
        w[4 * u + 1] = x.y;
        w[4 * u + 2] = x.z;
        w[4 * u + 3] = x.w;
      }
      tmem_st32(tmem + lane_off + kColQl + 32 * q, w);
    }
    if (!live) {
#pragma unroll
      for (int v = 0; v < 4; ++v) *(uint4*)(qrope + h * 64 + (v << 4)) = make_uint4(0, 0, 0, 0);
    }
    fence_proxy_async_smem();  // visible to the MMA (async proxy)
    tmem_st_wait();
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(q_ready);
  }
  pdl_wait();        // the selected positions come from the previous kernel
  // Cache row of every selected position of this split (-1: padding or invalid), while
  // Q is in flight; all index loads of a thread are in flight together, then all
  // page-table loads.
  {
    constexpr int kPer = (kMaxSplitLen + kThreads - 1) / kThreads;
    int pos[kPer];
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
      const int j = tid + u * kThreads;
      pos[u] = (j < n_tiles * kTok && j_begin + j < j_end) ? __ldg(p.idx + (int64_t)tok * p.top_k + j_begin + j)
                                                            : -1;
      if (pos[u] >= n_vis || pos[u] < -1) {
        if (c == 0) atomicOr(p.err, DSA_DEVERR_INDEX);
        pos[u] = -1;
      }
    }
    int pg[kPer];
#pragma unroll
    for (int u = 0; u < kPer; ++u)
      pg[u] = pos[u] >= 0 ? __ldg(p.tv.block_table + (int64_t)b * p.tv.max_pages + (pos[u] >> 6)) : -1;
    int mylast = -1;
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
      const int j = tid + u * kThreads;
      if (j >= n_tiles * kTok) break;
      int rid = -1;
      if (pos[u] >= 0) {
        if (pg[u] < 0 || pg[u] >= p.tv.num_pages) {
          if (c == 0) atomicOr(p.err, DSA_DEVERR_PAGE_ID);
        } else {
          rid = pg[u] * kPage + (pos[u] & 63);
          mylast = j;
        }
      }
      rowid[j] = rid;
    }
    if (mylast >= 0) atomicMax(last_valid_s, mylast);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // a selected row stands in for empty slots; tiles past the last selected row (the
  // padding of rows shorter than K) are skipped, and a split without any selected row
  // attends to nothing
  int fill = -1;
  for (int j = 0; j < n_tiles * kTok && fill < 0; ++j) fill = rowid[j];
  const int last_valid = *last_valid_s;
  const int n_tiles_run = last_valid >= 0 ? last_valid / kTok + 1 : 0;
  cluster_wait();  // both CTAs' barriers exist before any remote traffic

  if (warp < kGatherWarps || warp >= kExtraWarp0) {
    // ============================ gather (TMA) =========================================
    // Per tile and per group g of 4 slots: four 128-byte pieces q = 0..3 of this CTA's
    // latent dims (128-byte swizzled rows) and the 64-byte piece q = 4 of its rope dims
    // (64-byte swizzled rows), each one gather4 of four rows.  Gather i = 5g + q of a
    // tile is issued by lane i / 7 of gather warp i % 7 (warps 0-2, then 16-19).  Empty slots fetch a selected row;
    // their logits are masked; warps 16-19 take gathers too (7 warps: issuing a gather
    // costs its warp ~50 ns, so the issue is spread).  (FP8: pieces q = 0, 1 of codes and
    // q = 2 of rope per group, i = 3g + q, by warps 0-2, whose remaining lanes copy the
    // rows' scales; warps 16-19 convert each tile once it has landed.)
    if constexpr (!FP8) {
      const int gw = warp < kGatherWarps ? warp : kGatherWarps + (warp - kExtraWarp0);  // 7 gather warps
      const int i = lane * (kGatherWarps + 4) + gw;
      const bool mine = i < kGathers;
      const int g = i / 5, q = i - 5 * (i / 5);
      const int x = q < 4 ? 256 * (int)c + 64 * q : 512 + 32 * (int)c;
      const uint32_t doff = q < 4 ? q * kRegion + g * 512 : 4 * kRegion + g * 256;
      const CUtensorMap* map = q < 4 ? &kvmap : &ropemap;
      const uint32_t my_bytes = __reduce_add_sync(0xffffffffu, mine ? (q < 4 ? 512u : 256u) : 0u);
      uint32_t armed = 0, armed_parity = 0;  // stages with gathers issued, and their phase parity
      for (int n = 0; n < n_tiles_run; ++n) {
        const int stage = n % kStages;
        bool good = true;
        if (lane == 0) {
          // stage buffers 2-3 hold Q until the sending warps have moved it to tensor memory
          if (n == 2) good = mbar_wait(q_ready, 0, abort_flag, p.err);
          if (good) good = mbar_wait(&kv_empty[stage], ((n / kStages) & 1) ^ 1, abort_flag, p.err);
          if (good) mbar_arrive_expect_tx(&kv_full[stage], my_bytes);
        }
        if (!__shfl_sync(0xffffffffu, good, 0)) break;
        __syncwarp();
        armed |= 1u << stage;
        armed_parity = (armed_parity & ~(1u << stage)) | ((uint32_t)((n / kStages) & 1) << stage);
        if (mine) {
          const int4 v = *(const int4*)(rowid + n * kTok + 4 * g);
          tma_gather4(smem_u32(stages + stage * kStageBytes) + doff, map, &kv_full[stage], x,
                      v.x >= 0 ? v.x : fill, v.y >= 0 ? v.y : fill, v.z >= 0 ? v.z : fill, v.w >= 0 ? v.w : fill);
        }
      }
      // after an abort, let the gathers still in flight land before the CTA moves on (a
      // phase another warp never armed completes no more: the wait then ends at its limit)
      if (*abort_flag && lane == 0) {
        for (int st = 0; st < kStages; ++st) {
          if (!(armed >> st & 1)) continue;
          const long long t0 = clock64();
          while (!mbar_try_wait(smem_u32(&kv_full[st]), (armed_parity >> st) & 1) && clock64() - t0 < kWaitLimitCycles) {
          }
        }
      }
      __syncwarp();
    } else if (warp < kGatherWarps) {
      // FP8, issuers (warps 0-2, blocking waits): lane l of warp w takes item i = 3 l + w:
      // gather i (i < 48: pieces q = i % 3 of group i / 3), else the scale copies of rows
      // j = i - 48 and j + 48 (below 64)
      const int i = lane * kGatherWarps + warp;
      const bool gat = i < kGathersFp8;
      const int g = i / 3, q = i - 3 * (i / 3);
      const int x = q < 2 ? 256 * (int)c + 128 * q : 32 * (int)c;
      const uint32_t doff = q < 2 ? (2 + q) * kRegion + g * 512 : 4 * kRegion + g * 256;
      const CUtensorMap* map = q < 2 ? &kvmap : &ropemap;
      const int j0 = i - kGathersFp8;
      const uint32_t my_bytes = __reduce_add_sync(0xffffffffu, gat ? (q < 2 ? 512u : 256u) : 0u);
      uint32_t armed = 0, armed_parity = 0;  // stages with copies issued, and their phase parity
      for (int n = 0; n < n_tiles_run; ++n) {
        const int stage = n % kStages;
        bool good = true;
        if (lane == 0) {
          // stage buffers 2-3 hold Q until the sending warps have moved it to tensor memory
          if (n == 2) good = mbar_wait(q_ready, 0, abort_flag, p.err);
          if (good) good = mbar_wait(&kv_empty[stage], ((n / kStages) & 1) ^ 1, abort_flag, p.err);
          if (good) mbar_arrive_expect_tx(&kv_full[stage], my_bytes);
        }
        if (!__shfl_sync(0xffffffffu, good, 0)) break;
        __syncwarp();
        armed |= 1u << stage;
        armed_parity = (armed_parity & ~(1u << stage)) | ((uint32_t)((n / kStages) & 1) << stage);
        if (gat) {
          const int4 v = *(const int4*)(rowid + n * kTok + 4 * g);
          tma_gather4(smem_u32(stages + stage * kStageBytes) + doff, map, &kv_full[stage], x, v.x >= 0 ? v.x : fill,
                      v.y >= 0 ? v.y : fill, v.z >= 0 ? v.z : fill, v.w >= 0 ? v.w : fill);
        } else {
          for (int r = j0; r < kTok; r += kScaleLanes) {
            const int rid = rowid[n * kTok + r];
            cp_async16(smem_u32(scale_area + stage * (kTok * 4) + r * 4),
                       p.kv_scale + (int64_t)(rid >= 0 ? rid : fill) * 4);
          }
          cp_async_arrive_noinc(&kv_full[stage]);
        }
      }
      // nothing may still be landing in shared memory once the CTA moves on (on the normal
      // path these phases completed long ago)
      if (lane == 0) {
        for (int st = 0; st < kStages; ++st) {
          if (!(armed >> st & 1)) continue;
          const long long t0 = clock64();
          while (!mbar_try_wait(smem_u32(&kv_full[st]), (armed_parity >> st) & 1) && clock64() - t0 < kWaitLimitCycles) {
          }
        }
      }
      __syncwarp();
    } else {
      // FP8, converters (warps 16-19, blocking waits): tile m once its rows have landed,
      // rows [8 pp, 8 pp + 8) of the passes pp = warp - 16, warp - 12; lane = 4 * (row
      // within the pass) + output piece
      const int qo = lane & 3, piece = qo >> 1, half = qo & 1;
      for (int m = 0; m < n_tiles_run; ++m) {
        const int stage = m % kStages;
        bool ok = true;
        if (lane == 0) ok = mbar_wait(&kv_full[stage], (m / kStages) & 1, abort_flag, p.err);
        if (!__shfl_sync(0xffffffffu, ok, 0)) break;
        __syncwarp();
        uint8_t* st = stages + stage * kStageBytes;
        const float* sca = scale_area + stage * (kTok * 4);
        for (int pp = warp - kExtraWarp0; pp < kTok / 8; pp += kConvWarps) {
          const int r = 8 * pp + (lane >> 2);
          const uint32_t sw = (uint32_t)(r & 7);
          const uint8_t* raw = st + (2 + piece) * kRegion + r * 128;
          uint4 in[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) in[u] = *(const uint4*)(raw + ((((uint32_t)(4 * half + u)) ^ sw) << 4));
          const float sc60 = sca[r * 4 + 2 * (int)c + piece] * 0x1p60f;  // exact: a power-of-two factor
          const uint32_t sc2 = pack_bf16x2(sc60, sc60);
          __syncwarp();  // every lane has read its codes before any piece of its row is overwritten
          uint8_t* out = st + qo * kRegion + r * 128;
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            uint32_t o[8];
            e4m3x16_scaled_to_bf16(in[u], sc2, o);
            *(uint4*)(out + ((((uint32_t)(2 * u)) ^ sw) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
            *(uint4*)(out + ((((uint32_t)(2 * u + 1)) ^ sw) << 4)) = make_uint4(o[4], o[5], o[6], o[7]);
          }
          __syncwarp();
        }
        fence_proxy_async_smem();  // the MMAs read the rows (async proxy)
        __syncwarp();
        if (lane == 0) mbar_arrive(&kv_conv[stage]);
      }
    }
  } else if (warp == kMmaWarp) {
    // ============================ MMA issuer ==========================================
    // Event driven: the logits of tile t (QK(t): needs its rows, and its logit buffer
    // t & 1 back from tile t - 2, whose logits the softmax has read) and P.V of tile m
    // (needs P(m)) are issued as soon as their inputs are ready, so neither waits behind
    // the other.  QK(t) contracts the 288 own dims: 16 latent steps
    // (A = Q latent columns in tensor memory) and 2 rope steps (A = Q rope in shared
    // memory, B = this CTA's 32 of the 64 gathered rope dims).
    // The whole warp runs the loop (operands and decisions stay warp-uniform); one
    // elected lane issues every MMA and commit, so each commit tracks all of them.
    {
      const uint32_t id_qk = idesc(128, kTok, 1u, 1u);
      const uint32_t id_pv = idesc_bmn(128, 256, 1u, 1u);
      const uint32_t qr = smem_u32(qrope);
      const bool leader = elect_one();
      bool ok = true;
      if (lane == 0) ok = mbar_wait(q_ready, 0, abort_flag, p.err);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      int next_qk = 0, next_pv = 0;
      long long idle_since = clock64();
      while (ok && next_pv < n_tiles_run) {
        bool progress = false;
        if (next_qk < n_tiles_run) {
          const int t = next_qk, stage = t % kStages, b = t & 1;
          bool ready = false;
          if (lane == 0)
            ready = mbar_test(smem_u32(FP8 ? &kv_conv[stage] : &kv_full[stage]), (t / kStages) & 1) &&
                    (t < 2 || mbar_test(smem_u32(&s_free[b]), ((t - 2) >> 1) & 1));
          if (__shfl_sync(0xffffffffu, ready, 0)) {
            tc_fence_after();
            const uint32_t sb = smem_u32(stages + stage * kStageBytes);
            const uint32_t d = tmem + kColS + 64 * b;
            if (leader) {
#pragma unroll
              for (int k = 0; k < 16; ++k)
                mma_f16_ts(d, tmem + kColQl + 8 * k, desc_sw128(sb + (k >> 2) * kRegion + (k & 3) * 32), id_qk, k > 0);
#pragma unroll
              for (int k = 0; k < 2; ++k)
                mma_f16(d, desc_sw64(qr + 32 * k), desc_sw64(sb + 4 * kRegion + 32 * k), id_qk, 1u);
              tc_commit(&s_full[b]);
            }
            __syncwarp();
            ++next_qk;
            progress = true;
          }
        }
        if (next_pv < next_qk) {
          bool ready = false;
          if (lane == 0) ready = mbar_test(smem_u32(&p_full[next_pv & 1]), (next_pv >> 1) & 1);
          if (__shfl_sync(0xffffffffu, ready, 0)) {
            const int m = next_pv, stage = m % kStages;
            tc_fence_after();
            const uint32_t sb = smem_u32(stages + stage * kStageBytes);
            const uint32_t pb = smem_u32(xch + (m & 1) * kXchBytes);
            if (leader) {
#pragma unroll
              for (int j = 0; j < kTok / 16; ++j)
                mma_f16(tmem + kColO, desc_sw128(pb + 32 * j), desc_sw128_mn(sb + j * 2048, kRegion, 1024), id_pv,
                        (m > 0 || j > 0) ? 1u : 0u);
              tc_commit(&pv_done[m & 1]);
              tc_commit(&kv_empty[stage]);
              tc_commit_mc(&xch_empty[m & 1], (uint16_t)(1u << peer));  // the peer may send tile m + 2
            }
            __syncwarp();
            ++next_pv;
            progress = true;
          }
        }
        if (progress) {
          idle_since = clock64();
        } else {
          bool quit = false;
          if (lane == 0) {
            if (*abort_flag) {
              quit = true;
            } else if (clock64() - idle_since > kWaitLimitCycles) {
              atomicOr(p.err, DSA_DEVERR_TIMEOUT);
              *abort_flag = 1;
              quit = true;
            }
          }
          if (__shfl_sync(0xffffffffu, quit, 0)) ok = false;
        }
      }
      if (leader) {
        tc_commit(drain);
        const long long t0 = clock64();
        while (!mbar_try_wait(smem_u32(drain), 0) && clock64() - t0 < kWaitLimitCycles) {
        }
      }
      __syncwarp();
    }
  } else if (warp < kFinWarp0) {
    // ============================ senders =============================================
    // Per tile t: load this CTA's partial logits, scale them by softmax_scale * log2(e)
    // and round them to fp16 (both CTAs sum the same rounded halves, so their softmax is
    // identical), stage them and send them (one bulk copy per warp) to the peer's receive
    // buffer t & 1 once the peer is done with tile t - 2 there.  (The finishing warps
    // derive the same rounded values from the logits themselves.)  Every wait is bounded.
    const int quarter = warp & 3;
    const int h = quarter * 32 + lane;  // head row == TMEM lane
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const uint32_t warp_rows = (uint32_t)(quarter * 32) * (kTok * 2);  // this warp's 4 KB slice
    const uint32_t xch_peer0 = map_to_rank(smem_u32(xch) + warp_rows, peer);
    const uint32_t xfull_peer0 = map_to_rank(smem_u32(&xch_full[0]), peer);
    const uint32_t myrow = (uint32_t)h * (kTok * 2);
    const uint32_t sw = (uint32_t)(h & 7);
    for (int t = 0; t < n_tiles_run; ++t) {
      const int bb = t & 1;
      bool good = true;
      if (lane == 0) good = mbar_wait(&s_full[bb], (t >> 1) & 1, abort_flag, p.err);
      if (!__shfl_sync(0xffffffffu, good, 0)) break;
      __syncwarp();
      tc_fence_after();
      uint32_t dst[kTok / 2];
      {
        uint32_t v0[32], v1[32];
        tmem_ld32(tmem + lane_off + kColS + 64 * bb, v0);
        tmem_ld32(tmem + lane_off + kColS + 64 * bb + 32, v1);
        tmem_ld_wait();
        const uint64_t sc2 = f2_pack(p.scale_log2, p.scale_log2);
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          float a0, a1, b0, b1;
          f2_unpack(f2_mul(f2_pack(__uint_as_float(v0[2 * j]), __uint_as_float(v0[2 * j + 1])), sc2), a0, a1);
          f2_unpack(f2_mul(f2_pack(__uint_as_float(v1[2 * j]), __uint_as_float(v1[2 * j + 1])), sc2), b0, b1);
          dst[j] = cvt_f16x2(a0, a1);
          dst[16 + j] = cvt_f16x2(b0, b1);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&s_free[bb]);
        if (t > 0) bulk_wait_read0();  // the staging is free once the copy of tile t - 1 read it
      }
      __syncwarp();
      uint8_t* sbuf = stg;
#pragma unroll
      for (int u = 0; u < kTok / 8; ++u)
        *(uint4*)(sbuf + myrow + (((uint32_t)u ^ sw) << 4)) =
            make_uint4(dst[4 * u], dst[4 * u + 1], dst[4 * u + 2], dst[4 * u + 3]);
      fence_proxy_async_smem();  // the bulk copy reads it (async proxy)
      __syncwarp();
      if (lane == 0) {
        if (t >= 2) good = mbar_wait_cluster(&xch_empty[bb], ((t >> 1) & 1) ^ 1, abort_flag, p.err);
        if (good) {
          bulk_copy_to_peer(xch_peer0 + bb * kXchBytes, smem_u32(sbuf) + warp_rows, 32 * kTok * 2,
                            xfull_peer0 + bb * 8);
          bulk_commit();
        }
      }
      if (!__shfl_sync(0xffffffffu, good, 0)) break;
    }
  } else {
    // ============================ finishers + epilogue ================================
    const int quarter = warp & 3;
    const int h = quarter * 32 + lane;  // head row == TMEM lane
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const uint32_t myrow = (uint32_t)h * (kTok * 2);
    const uint32_t sw = (uint32_t)(h & 7);
    float m_ref = -INFINITY, l = 0.f;
    bool ok = true;

    // Finishing: the two warps of a row quarter take key columns [32 hf, 32 hf + 32) of
    // each tile (hf = 0: warps 8-11, hf = 1: warps 12-15).  Each rounds its own half of
    // the logits exactly as the senders do, adds the peer's half, and the pair meets once
    // per tile to share the row maxima (so both keep the same reference maximum); each
    // keeps its half of the row sum, stores its half of P and rescales half of O.  Both
    // warps run every tile and reach the pair's barrier whatever happened, so a wait that
    // gives up never strands the partner; a failed wait skips the work.
    const int hf = warp >= kFinWarpB0 ? 1 : 0;
    const uint64_t sc2 = f2_pack(p.scale_log2, p.scale_log2);
    bool good = true;
    for (int n = 0; n < n_tiles_run; ++n) {
      const int bb = n & 1;
      const uint32_t vmask = __ballot_sync(0xffffffffu, rowid[n * kTok + 32 * hf + lane] >= 0);
      if (lane == 0 && good) {
        good = mbar_wait(&xch_full[bb], (n >> 1) & 1, abort_flag, p.err);
        if (good && hf == 0 && h == 0 && n + 2 < n_tiles_run)  // one thread re-arms it for tile n + 2
          mbar_arrive_expect_tx(&xch_full[bb], kXchBytes);
        if (good) good = mbar_wait(&s_full[bb], (n >> 1) & 1, abort_flag, p.err);
      }
      good = __shfl_sync(0xffffffffu, good, 0);
      __syncwarp();
      float s[32];  // scaled logits of this warp's half of tile n
      float lmax = -INFINITY;
      if (good) {
        tc_fence_after();
        uint32_t v[32];
        tmem_ld32(tmem + lane_off + kColS + 64 * bb + 32 * hf, v);
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&s_free[bb]);
        const uint8_t* recv = xch + bb * kXchBytes + myrow;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const uint4 r = *(const uint4*)(recv + ((((uint32_t)(4 * hf + u)) ^ sw) << 4));
          const uint32_t rr[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int jj = 8 * u + 2 * e;
            float a0, a1;
            f2_unpack(f2_mul(f2_pack(__uint_as_float(v[jj]), __uint_as_float(v[jj + 1])), sc2), a0, a1);
            f16x2_to_f32(rr[e], s[jj], s[jj + 1]);
            add_f16x2_to(cvt_f16x2(a0, a1), s[jj], s[jj + 1]);  // the same rounded half the peer got
          }
        }
        if (vmask != 0xffffffffu) {
#pragma unroll
          for (int jj = 0; jj < 32; ++jj) s[jj] = ((vmask >> jj) & 1u) ? s[jj] : -INFINITY;
        }
        float mx[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) mx[e] = max3f(s[e], s[8 + e], fmaxf(s[16 + e], s[24 + e]));
        lmax = max3f(max3f(mx[0], mx[1], mx[2]), max3f(mx[3], mx[4], mx[5]), fmaxf(mx[6], mx[7]));
      }
      maxx[(bb * 2 + hf) * 128 + h] = lmax;
      named_bar_sync(2 + quarter, 64);
      const float pmax = maxx[(bb * 2 + (hf ^ 1)) * 128 + h];
      if (!good) continue;
      const float tmax = fmaxf(lmax, pmax);
      float alpha = 1.f;
      bool rescale = false;
      if (tmax != -INFINITY && (m_ref == -INFINITY || tmax > m_ref + 8.f)) {
        if (m_ref != -INFINITY) {
          alpha = fast_exp2(m_ref - tmax);
          rescale = true;
        }
        m_ref = tmax;
      }
      const float msub = m_ref == -INFINITY ? 0.f : m_ref;  // nothing visible yet: all weights 0
      const uint64_t negm = f2_pack(-msub, -msub);
      uint64_t ps[4] = {0ull, 0ull, 0ull, 0ull};  // paired partial sums
      uint32_t pw[16];
#pragma unroll
      for (int jj = 0; jj < 16; ++jj) {
        float x0, x1;
        f2_unpack(f2_add(f2_pack(s[2 * jj], s[2 * jj + 1]), negm), x0, x1);
        x0 = fast_exp2(x0);  // 2^-inf = 0 for masked positions
        x1 = fast_exp2(x1);
        ps[jj & 3] = f2_add(ps[jj & 3], f2_pack(x0, x1));
        pw[jj] = cvt_bf16x2(x0, x1);
      }
      float r0, r1, r2, r3;
      f2_unpack(f2_add(ps[0], ps[1]), r0, r1);
      f2_unpack(f2_add(ps[2], ps[3]), r2, r3);
      l = l * alpha + ((r0 + r2) + (r1 + r3));
      if (__any_sync(0xffffffffu, rescale)) {  // rare: move O (this warp's half of it) to the new reference
        if (n > 0) {  // ... once P.V(n - 1), the last one issued, has updated it
          bool g2 = true;
          if (lane == 0) g2 = mbar_wait(&pv_done[(n - 1) & 1], ((n - 1) >> 1) & 1, abort_flag, p.err);
          good = __shfl_sync(0xffffffffu, g2, 0);
          __syncwarp();
          tc_fence_after();
        }
        if (good) {
#pragma unroll 1
          for (int ch = 4 * hf; ch < 4 * hf + 4; ++ch) {
            uint32_t v[32];
            tmem_ld32(tmem + lane_off + kColO + 32 * ch, v);
            tmem_ld_wait();
#pragma unroll
            for (int jj = 0; jj < 32; ++jj) v[jj] = __float_as_uint(__uint_as_float(v[jj]) * alpha);
            tmem_st32(tmem + lane_off + kColO + 32 * ch, v);
          }
        }
      }
      if (!good) continue;
      {  // this warp's half of row h of P(n), over the peer's data in the receive buffer
        uint8_t* prow = xch + bb * kXchBytes + myrow;
#pragma unroll
        for (int u = 0; u < 4; ++u)
          *(uint4*)(prow + ((((uint32_t)(4 * hf + u)) ^ sw) << 4)) =
              make_uint4(pw[4 * u], pw[4 * u + 1], pw[4 * u + 2], pw[4 * u + 3]);
      }
      fence_proxy_async_smem();  // visible to the MMA (async proxy)
      tmem_st_wait();            // (rescaled O)
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[bb]);
    }
    // the row sums' halves meet; warps 12-15 are done after this
    {
      float* lx = maxx + ((n_tiles_run & 1) * 2 + 1) * 128;  // a slot the last tile did not use
      if (hf) lx[h] = l;
      named_bar_sync(2 + quarter, 64);
      if (!hf) l += lx[h];
    }
    ok = good && !*abort_flag;
    if (!hf) {
    // ---- epilogue: O / l -> this CTA's 256 value dims ----------------------------------
    if (ok && n_tiles_run > 0) {
      if (lane == 0) ok = mbar_wait(&pv_done[(n_tiles_run - 1) & 1], ((n_tiles_run - 1) >> 1) & 1, abort_flag, p.err);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      __syncwarp();
    }
    tc_fence_after();
    const float inv = l > 0.f ? 1.f / l : 0.f;
    const bool live = h < H;
    if (p.n_splits == 1) {
      if (ok) {
#pragma unroll 1
        for (int ch = 0; ch < 8; ++ch) {
          uint32_t v[32];
          if (n_tiles_run > 0) {
            tmem_ld32(tmem + lane_off + kColO + 32 * ch, v);
            tmem_ld_wait();
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = 0u;
          }
          if (!live) continue;
          uint4* dst = (uint4*)(p.out + ((int64_t)tok * H + h) * kValueDim + 256 * (int)c + 32 * ch);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint4 w;
            w.x = pack_bf16x2(__uint_as_float(v[8 * q]) * inv, __uint_as_float(v[8 * q + 1]) * inv);
            w.y = pack_bf16x2(__uint_as_float(v[8 * q + 2]) * inv, __uint_as_float(v[8 * q + 3]) * inv);
            w.z = pack_bf16x2(__uint_as_float(v[8 * q + 4]) * inv, __uint_as_float(v[8 * q + 5]) * inv);
            w.w = pack_bf16x2(__uint_as_float(v[8 * q + 6]) * inv, __uint_as_float(v[8 * q + 7]) * inv);
            dst[q] = w;
          }
        }
      }
    } else if (p.sib_merge) {
      // Two splits in one cluster of four (rank 2 s + c: split s, value half c).  Split s
      // finalizes value columns [128 s, 128 s + 128) of this half: it hands the other 128
      // columns of its O (unnormalized) and every row's (m_ref, l) to its sibling (rank
      // ^ 2) through distributed shared memory and receives the sibling's in exchange.
      // The columns travel normalized (O / l, rounded to fp16: relative 2^-11, below the
      // bf16 rounding of the output) with (m_ref, l) in f32.  The (then idle) stage
      // buffers hold the outbox and the inbox: row h's 16-byte chunk u (8 columns) at
      // slot u ^ (h & 15) (conflict-free), then the 128 (m, l) pairs.
      const uint32_t sib = rank ^ 2u;
      const int s_me = (int)(rank >> 1);
      uint8_t* outbox = stages;
      uint8_t* inbox = stages + kSibBytes;
      if (h == 0) {
        mbar_arrive_expect_tx(m_full, kSibBytes);                // our inbox may fill from now on
        mbar_arrive_remote(map_to_rank(smem_u32(m_ready), sib));  // tell the sibling
      }
      const int send_col = 128 * (1 - s_me);
#pragma unroll 1
      for (int q = 0; q < 4; ++q) {
        uint32_t v[32];
        if (n_tiles_run > 0 && ok) {
          tmem_ld32(tmem + lane_off + kColO + send_col + 32 * q, v);
          tmem_ld_wait();
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] = 0u;
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const float* f = (const float*)v + 8 * u;
          *(uint4*)(outbox + h * 256 + (((4 * q + u) ^ (h & 15)) << 4)) =
              make_uint4(cvt_f16x2(f[0] * inv, f[1] * inv), cvt_f16x2(f[2] * inv, f[3] * inv),
                         cvt_f16x2(f[4] * inv, f[5] * inv), cvt_f16x2(f[6] * inv, f[7] * inv));
        }
      }
      ((float2*)(outbox + 128 * 256))[h] = make_float2(ok ? m_ref : -INFINITY, ok ? l : 0.f);
      fence_proxy_async_smem();  // the bulk copies read it (async proxy)
      __syncwarp();
      if (lane == 0 && mbar_wait_cluster(m_ready, 0, abort_flag, p.err)) {  // the sibling's inbox is free
        // this warp's 32 rows and their (m, l) pairs, one bulk copy each
        const uint32_t rows = (uint32_t)(quarter * 32);
        const uint32_t sib_full = map_to_rank(smem_u32(m_full), sib);
        bulk_copy_to_peer(map_to_rank(smem_u32(inbox) + rows * 256, sib), smem_u32(outbox) + rows * 256, 32 * 256,
                          sib_full);
        bulk_copy_to_peer(map_to_rank(smem_u32(inbox) + 128 * 256 + rows * 8, sib),
                          smem_u32(outbox) + 128 * 256 + rows * 8, 32 * 8, sib_full);
        bulk_commit();
      }
      bool good = true;
      if (lane == 0) good = mbar_wait(m_full, 0, abort_flag, p.err);
      good = __shfl_sync(0xffffffffu, good, 0);
      __syncwarp();
      if (good && ok) {  // (warp-uniform: the tensor-memory loads below take the whole warp)
        const float2 ms = ((const float2*)(inbox + 128 * 256))[h];  // the sibling's (m, l)
        const float m0 = s_me == 0 ? m_ref : ms.x, l0 = s_me == 0 ? l : ms.y;
        const float m1 = s_me == 0 ? ms.x : m_ref, l1 = s_me == 0 ? ms.y : l;
        const float mx = fmaxf(m0, m1);
        const float a0 = mx == -INFINITY || m0 == -INFINITY ? 0.f : exp2f(m0 - mx);
        const float a1 = mx == -INFINITY || m1 == -INFINITY ? 0.f : exp2f(m1 - mx);
        const float den = l0 * a0 + l1 * a1;
        const float inv2 = den > 0.f ? 1.f / den : 0.f;
        const float w0 = a0 * inv2, w1 = a1 * inv2;  // split 0's and split 1's weight
        const float w_me = s_me == 0 ? w0 : w1;                          // on this CTA's O
        const float w_sib = s_me == 0 ? w1 * l1 : w0 * l0;               // on the sibling's O / l
#pragma unroll 1
        for (int q = 0; q < 4; ++q) {
          uint32_t v[32];
          if (n_tiles_run > 0) {
            tmem_ld32(tmem + lane_off + kColO + 128 * s_me + 32 * q, v);
            tmem_ld_wait();
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = 0u;
          }
          if (!live) continue;
          uint4* dst = (uint4*)(p.out + ((int64_t)tok * H + h) * kValueDim + 256 * (int)c + 128 * s_me + 32 * q);
          uint32_t packed[16];
#pragma unroll
          for (int u = 0; u < 4; ++u) {  // 8 columns per chunk
            const uint4 r = *(const uint4*)(inbox + h * 256 + (((4 * q + u) ^ (h & 15)) << 4));
            const uint32_t rr[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              float y0, y1;
              f16x2_to_f32(rr[i], y0, y1);
              const float o0 = fmaf(y0, w_sib, __uint_as_float(v[8 * u + 2 * i]) * w_me);
              const float o1 = fmaf(y1, w_sib, __uint_as_float(v[8 * u + 2 * i + 1]) * w_me);
              packed[4 * u + i] = pack_bf16x2(o0, o1);
            }
          }
#pragma unroll
          for (int j = 0; j < 4; ++j)
            dst[j] = make_uint4(packed[4 * j], packed[4 * j + 1], packed[4 * j + 2], packed[4 * j + 3]);
        }
      }
    } else {
      // More than two splits: publish this split's part of the CTA's value half, O / l
      // (column-major, so the stores and the combine's loads are coalesced across heads)
      // and its log2-sum-exp.
      const int64_t half_id = ((int64_t)tok * p.n_splits + split) * 2 + c;
      if (ok) {
        const int HP = (H + 3) & ~3;  // head stride of the partials (16-byte rows for the combine)
        float* po = p.part_o + half_id * 256 * HP;
#pragma unroll 1
        for (int ch = 0; ch < 8; ++ch) {
          uint32_t v[32];
          if (n_tiles_run > 0) {
            tmem_ld32(tmem + lane_off + kColO + 32 * ch, v);
            tmem_ld_wait();
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = 0u;
          }
          if (!live) continue;
#pragma unroll
          for (int j = 0; j < 32; ++j) po[(32 * ch + j) * HP + h] = __uint_as_float(v[j]) * inv;
        }
        if (live) p.part_lse[half_id * HP + h] = l > 0.f ? m_ref + __log2f(l) : -INFINITY;
      }
      // sfa_combine_kernel (the next launch) merges the splits of every (token, half)
    }
    }  // the first finishing warp of each row quarter
  }

  // ---- tear-down ---------------------------------------------------------------------
  if (warp > kMmaWarp && lane == 0) bulk_wait_read0();
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // the peer's last remote arrivals and stores have landed
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// Merge of more than two splits: out[tok, h, 256 c + col] = sum_s w_s O_s / l_s with
// w_s = 2^(lse_s - max) / sum 2^(lse - max), the splits taken in order (the result does
// not depend on which CTA finished first).  One CTA of 128 threads per (token, value
// half, 8-column chunk); thread t takes heads 4 (t % 32) .. + 3 and columns 2 (t / 32)
// .. + 1 of the chunk: 16-byte loads over 4 heads (the partials are column-major, their
// head stride H rounded up to a multiple of 4).  Every split's log2-sum-exp and the
// values of up to eight splits are in flight together: a merge of eight splits waits
// for one round of loads.
constexpr int kCombineCols = 8;
constexpr int kCombineThreads = 128;
constexpr int kCombineGroup = 8;       // splits whose value loads are in flight together
constexpr int kMaxCombineSplits = 16;  // (the planner makes at most 16 splits)

__global__ void __launch_bounds__(kCombineThreads) sfa_combine_kernel(SfaParams p) {
  pdl_trigger();
  pdl_wait();  // the partials of the attention kernel
  constexpr int kChunks = 256 / kCombineCols;
  const int tok = blockIdx.y, c = blockIdx.x / kChunks, k = blockIdx.x % kChunks;
  const int H = p.n_heads, S = p.n_splits, HP = (H + 3) & ~3;  // partials' head stride
  const int h0 = 4 * (threadIdx.x & 31), col0 = kCombineCols * k + 2 * (threadIdx.x >> 5);
  if (h0 >= H) return;
  const int64_t base = (int64_t)tok * S * 2 + c;  // + 2 s: split s of this half
  float4 lse[kMaxCombineSplits];
#pragma unroll
  for (int s2 = 0; s2 < kMaxCombineSplits; ++s2)
    if (s2 < S) lse[s2] = *(const float4*)(p.part_lse + (base + 2 * s2) * HP + h0);
  float acc[2][4] = {};  // [column][head]
  float wsum[4] = {0.f, 0.f, 0.f, 0.f};
  float4 mx = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
  auto wt = [](float l, float m) { return m != -INFINITY ? exp2f(l - m) : 0.f; };
#pragma unroll 1
  for (int s0 = 0; s0 < S; s0 += kCombineGroup) {
    float4 v[kCombineGroup][2];
#pragma unroll
    for (int u = 0; u < kCombineGroup; ++u) {
      const float* po = p.part_o + ((base + 2 * min(s0 + u, S - 1)) * 256 + col0) * HP + h0;
      v[u][0] = *(const float4*)po;
      v[u][1] = *(const float4*)(po + HP);
    }
    if (s0 == 0) {  // (the first group's values are in flight meanwhile)
#pragma unroll
      for (int s2 = 0; s2 < kMaxCombineSplits; ++s2)
        if (s2 < S)
          mx = make_float4(fmaxf(mx.x, lse[s2].x), fmaxf(mx.y, lse[s2].y), fmaxf(mx.z, lse[s2].z),
                           fmaxf(mx.w, lse[s2].w));
    }
#pragma unroll
    for (int u = 0; u < kCombineGroup; ++u) {
      if (s0 + u >= S) break;
      float4 l = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int s2 = 0; s2 < kMaxCombineSplits; ++s2)
        if (s2 == s0 + u) l = lse[s2];
      const float w[4] = {wt(l.x, mx.x), wt(l.y, mx.y), wt(l.z, mx.z), wt(l.w, mx.w)};
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        acc[j][0] += w[0] * v[u][j].x;
        acc[j][1] += w[1] * v[u][j].y;
        acc[j][2] += w[2] * v[u][j].z;
        acc[j][3] += w[3] * v[u][j].w;
      }
#pragma unroll
      for (int e = 0; e < 4; ++e) wsum[e] += w[e];
    }
  }
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    if (h0 + e >= H) break;  // heads past H in the last group of four (padding, never written)
    const float winv = wsum[e] > 0.f ? 1.f / wsum[e] : 0.f;
    uint32_t* dst = (uint32_t*)(p.out + ((int64_t)tok * H + h0 + e) * kValueDim + 256 * c + col0);
    *dst = pack_bf16x2(acc[0][e] * winv, acc[1][e] * winv);
  }
}

}  // namespace

cudaError_t launch_sfa_combine(const SfaParams& p, cudaStream_t s) {
  return launch_pdl(sfa_combine_kernel, dim3(2 * (256 / kCombineCols), p.tv.n_tokens), dim3(kCombineThreads), 0, s,
                    p);
}

cudaError_t launch_sfa_tc(const SfaParams& p, cudaStream_t s) {
  // the latent cache as [pages * 64 rows, 576]: one-row boxes of 64 elements (latent
  // pieces, 128-byte swizzle) and of 32 elements (rope pieces, 64-byte swizzle); FP8:
  // codes as [pages * 64, 512] with one-row boxes of 128 bytes, rope as [pages * 64, 64]
  CUtensorMap kvmap, ropemap;
  // Q as [tokens * heads, 576]: boxes of one token's heads, 64 elements (latent, 128-byte
  // swizzle) and 32 elements (rope, 64-byte swizzle) wide
  CUtensorMap qmap, qropemap;
  const uint64_t rows = (uint64_t)p.tv.num_pages * kPage;
  const bool fp8 = p.kv_codes != nullptr;
  const bool kv_ok = fp8 ? make_tma_2d_sw128(&kvmap, p.kv_codes, rows, 1, kValueDim, 1, false) &&
                               make_tma_2d_sw64_rows(&ropemap, p.kv_rope, rows, 2, kLatentDim - kValueDim)
                         : make_tma_2d_sw128(&kvmap, p.kv, rows, 2, kLatentDim, 1, false) &&
                               make_tma_2d_sw64_rows(&ropemap, p.kv, rows, 2, kLatentDim);
  if (!kv_ok ||
      !make_tma_2d_sw128(&qmap, p.q, (uint64_t)p.tv.n_tokens * p.n_heads, 2, kLatentDim, p.n_heads, false) ||
      !make_tma_2d_sw64_rows(&qropemap, p.q, (uint64_t)p.tv.n_tokens * p.n_heads, 2, kLatentDim, p.n_heads))
    return cudaErrorInvalidValue;
  auto kernel = fp8 ? sfa_tc_kernel<true> : sfa_tc_kernel<false>;
  const int smem = fp8 ? kSmemFp8 : kSmem;
  static std::atomic<int> smem_set[2][kMaxDevices];
  cudaError_t e = set_smem_once(kernel, smem, smem_set[fp8 ? 1 : 0]);
  if (e != cudaSuccess) return e;
  dim3 grid(2 * p.n_splits, p.tv.n_tokens);
  return launch_pdl_cluster(kernel, grid, dim3(kThreads), smem, s, p.sib_merge ? 4u : 2u, kvmap, ropemap, qmap,
                            qropemap, p);
}

}  // namespace dsa
