// Sparse Flash Attention over the positions the indexer selected.
//
// "Adapting and Optimizing Inference for a New Model Architecture on Ascend", section
// 3.1: the sparse attention reads the main-attention KV entries of the selected indices
// only and attends over that subset; "Inference Acceleration for Next-Gen Attention
// Architectures", section 3.2: the indices are non-contiguous, so rows are fetched by
// paged addressing and gathered.  DSA builds on MLA ("Day0 Inference Optimization on
// Ascend CANN", section 1): all heads share one 576-wide latent row per position, used
// whole as the key and, cut to its leading 512 entries, as the value.
//
// Baseline version on warp-level MMA (mma.sync m16n8k16, bf16 in, f32 accumulate):
// CTA = (split of the index list, block of 64 heads, query token), 8 warps; warp
// (g, v) owns heads 16g..16g+15 and value dims 256v..256v+255.  Per 64-position tile
// the selected rows are gathered with 16-byte cp.async into an XOR-swizzled shared tile
// (double buffered), logits and an online softmax (base-2, running max and sum) are
// kept in registers, and P.V accumulates in registers.  Splits write normalised partial
// outputs and their log-sum-exp; a combine kernel merges them.
#include "common.cuh"

namespace dsa {

namespace {

constexpr int kSfaThreads = 256;
constexpr int kHB = 64;           // heads per CTA
constexpr int kTile = 64;         // selected positions per tile
constexpr int kRowBytes = kLatentDim * 2;   // 1152
constexpr int kRowChunks = kRowBytes / 16;  // 72
constexpr int kTileBytes = kTile * kRowBytes;
constexpr int kQBytes = kHB * kRowBytes;
constexpr int kSfaSmem = kQBytes + 2 * kTileBytes + 2 * kTile * (int)sizeof(int64_t);

// Byte offset of 16-byte chunk c of row r in a [rows][72 chunks] tile; the low three
// chunk bits are XOR-ed with the row so that 8 rows of one column hit 8 bank groups.
__device__ __forceinline__ uint32_t swz(int r, int c) {
  return (uint32_t)(r * kRowBytes + (((c & ~7) | ((c ^ r) & 7)) << 4));
}

__global__ void __launch_bounds__(kSfaThreads, 1) sfa_mma_kernel(SfaParams p) {
  const int split = blockIdx.x, hb = blockIdx.y, tok = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int hg = warp & 3, vh = warp >> 2;
  const int H = p.n_heads;
  const int h0 = hb * kHB;
  int b, n_vis;
  resolve_token(p.tv, tok, &b, &n_vis, nullptr);

  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* Qs = smem;
  uint8_t* KVs = smem + kQBytes;
  int64_t* vrow = (int64_t*)(smem + kQBytes + 2 * kTileBytes);  // [2][64] cache row or -1

  const int j_begin = split * p.split_len;
  const int j_end = min(p.top_k, j_begin + p.split_len);
  const int n_tiles = j_end > j_begin ? (j_end - j_begin + kTile - 1) / kTile : 0;

  for (int c = tid; c < kHB * kRowChunks; c += kSfaThreads) {
    const int r = c / kRowChunks, ch = c % kRowChunks;
    const int h = h0 + r;
    const uint16_t* src = p.q + ((int64_t)tok * H + (h < H ? h : 0)) * kLatentDim + ch * 8;
    cp_async_16(smem_u32(Qs + swz(r, ch)), src, h < H ? 16 : 0);
  }

  auto load_tile = [&](int tile, int buf) {
    if (tid < kTile) {
      const int j = j_begin + tile * kTile + tid;
      int64_t rowid = -1;
      if (j < j_end) {
        const int pos = __ldg(p.idx + (int64_t)tok * p.top_k + j);
        if (pos >= n_vis || pos < -1) {
          atomicOr(p.err, DSA_DEVERR_INDEX);
        } else if (pos >= 0) {
          const int pg = physical_page(p.tv, b, pos >> 6, p.err);
          if (pg >= 0) rowid = (int64_t)pg * kPage + (pos & 63);
        }
      }
      vrow[buf * kTile + tid] = rowid;
    }
    __syncthreads();
    uint8_t* dst = KVs + buf * kTileBytes;
    for (int c = tid; c < kTile * kRowChunks; c += kSfaThreads) {
      const int r = c / kRowChunks, ch = c % kRowChunks;
      const int64_t rowid = vrow[buf * kTile + r];
      const uint16_t* src = p.kv + (rowid >= 0 ? rowid : 0) * kLatentDim + ch * 8;
      cp_async_16(smem_u32(dst + swz(r, ch)), src, rowid >= 0 ? 16 : 0);
    }
  };

  if (n_tiles > 0) load_tile(0, 0);
  cp_async_commit();

  const bool active = h0 + hg * 16 < H;
  float o[32][4];
#pragma unroll
  for (int i = 0; i < 32; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;

  for (int n = 0; n < n_tiles; ++n) {
    const int buf = n & 1;
    if (n + 1 < n_tiles) load_tile(n + 1, buf ^ 1);
    cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();
    if (active) {
      const uint8_t* kv = KVs + buf * kTileBytes;
      const int64_t* vr = vrow + buf * kTile;
      // ---- logits S[16 heads][64 positions] = Q . KV^T over 576 dims
      float s[8][4];
#pragma unroll
      for (int i = 0; i < 8; ++i) s[i][0] = s[i][1] = s[i][2] = s[i][3] = 0.f;
      const int mi = lane >> 3;
#pragma unroll 2
      for (int kk = 0; kk < kLatentDim / 16; ++kk) {
        uint32_t a[4];
        ldsm_x4(smem_u32(Qs + swz(hg * 16 + (mi & 1) * 8 + (lane & 7), 2 * kk + (mi >> 1))),
                a[0], a[1], a[2], a[3]);
#pragma unroll
        for (int np = 0; np < 4; ++np) {
          uint32_t bb[4];
          ldsm_x4(smem_u32(kv + swz(np * 16 + (mi >> 1) * 8 + (lane & 7), 2 * kk + (mi & 1))),
                  bb[0], bb[1], bb[2], bb[3]);
          mma_bf16_16816(s[2 * np], a, bb);
          mma_bf16_16816(s[2 * np + 1], a, bb + 2);
        }
      }
      // ---- online softmax in base 2
      float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int col = nt * 8 + (lane & 3) * 2 + (e & 1);
          const float v = vr[col] >= 0 ? s[nt][e] * p.scale_log2 : -INFINITY;
          s[nt][e] = v;
          if (e < 2) mx0 = fmaxf(mx0, v); else mx1 = fmaxf(mx1, v);
        }
      }
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
      const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
      const float ms0 = mn0 == -INFINITY ? 0.f : mn0, ms1 = mn1 == -INFINITY ? 0.f : mn1;
      const float al0 = exp2f(m0 - ms0), al1 = exp2f(m1 - ms1);
      m0 = mn0;
      m1 = mn1;
      float rs0 = 0.f, rs1 = 0.f;
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
        s[nt][0] = exp2f(s[nt][0] - ms0);
        s[nt][1] = exp2f(s[nt][1] - ms0);
        s[nt][2] = exp2f(s[nt][2] - ms1);
        s[nt][3] = exp2f(s[nt][3] - ms1);
        rs0 += s[nt][0] + s[nt][1];
        rs1 += s[nt][2] + s[nt][3];
      }
      l0 = l0 * al0 + rs0;
      l1 = l1 * al1 + rs1;
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        o[i][0] *= al0;
        o[i][1] *= al0;
        o[i][2] *= al1;
        o[i][3] *= al1;
      }
      // ---- O[16 heads][256 dims] += P[16][64] . V[64][256]
#pragma unroll
      for (int kk = 0; kk < kTile / 16; ++kk) {
        uint32_t a[4];
        a[0] = pack_bf16x2(s[2 * kk][0], s[2 * kk][1]);
        a[1] = pack_bf16x2(s[2 * kk][2], s[2 * kk][3]);
        a[2] = pack_bf16x2(s[2 * kk + 1][0], s[2 * kk + 1][1]);
        a[3] = pack_bf16x2(s[2 * kk + 1][2], s[2 * kk + 1][3]);
#pragma unroll
        for (int np = 0; np < 16; ++np) {
          uint32_t bb[4];
          ldsm_x4_t(smem_u32(kv + swz(kk * 16 + (mi & 1) * 8 + (lane & 7),
                                      (vh * 256 + np * 16) / 8 + (mi >> 1))),
                    bb[0], bb[1], bb[2], bb[3]);
          mma_bf16_16816(o[2 * np], a, bb);
          mma_bf16_16816(o[2 * np + 1], a, bb + 2);
        }
      }
    }
    __syncthreads();
  }
  cp_async_wait<0>();

  if (!active) return;
  l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
  const float inv0 = l0 > 0.f ? 1.f / l0 : 0.f, inv1 = l1 > 0.f ? 1.f / l1 : 0.f;
  const int hr0 = h0 + hg * 16 + (lane >> 2), hr1 = hr0 + 8;
  const int dcol = vh * 256 + (lane & 3) * 2;
  if (p.n_splits == 1) {
#pragma unroll
    for (int nt = 0; nt < 32; ++nt) {
      if (hr0 < H)
        *(uint32_t*)(p.out + ((int64_t)tok * H + hr0) * kValueDim + dcol + nt * 8) =
            pack_bf16x2(o[nt][0] * inv0, o[nt][1] * inv0);
      if (hr1 < H)
        *(uint32_t*)(p.out + ((int64_t)tok * H + hr1) * kValueDim + dcol + nt * 8) =
            pack_bf16x2(o[nt][2] * inv1, o[nt][3] * inv1);
    }
  } else {
    const int64_t base = ((int64_t)tok * p.n_splits + split) * H;
#pragma unroll
    for (int nt = 0; nt < 32; ++nt) {
      if (hr0 < H)
        *(float2*)(p.part_o + (base + hr0) * kValueDim + dcol + nt * 8) =
            make_float2(o[nt][0] * inv0, o[nt][1] * inv0);
      if (hr1 < H)
        *(float2*)(p.part_o + (base + hr1) * kValueDim + dcol + nt * 8) =
            make_float2(o[nt][2] * inv1, o[nt][3] * inv1);
    }
    if (vh == 0 && (lane & 3) == 0) {
      if (hr0 < H) p.part_lse[base + hr0] = l0 > 0.f ? m0 + __log2f(l0) : -INFINITY;
      if (hr1 < H) p.part_lse[base + hr1] = l1 > 0.f ? m1 + __log2f(l1) : -INFINITY;
    }
  }
}

// out[t, h, :] = sum_s 2^(lse_s - max) o_s / sum_s 2^(lse_s - max); 0 if no split had mass.
__global__ void __launch_bounds__(128) sfa_combine_kernel(SfaParams p) {
  const int h = blockIdx.x, tok = blockIdx.y;
  const int H = p.n_heads, S = p.n_splits;
  const int64_t base = (int64_t)tok * S * H;
  float mx = -INFINITY;
  for (int s = 0; s < S; ++s) mx = fmaxf(mx, p.part_lse[base + (int64_t)s * H + h]);
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float wsum = 0.f;
  if (mx != -INFINITY) {
    for (int s = 0; s < S; ++s) {
      const float w = exp2f(p.part_lse[base + (int64_t)s * H + h] - mx);
      const float4 v = *(const float4*)(p.part_o + (base + (int64_t)s * H + h) * kValueDim + threadIdx.x * 4);
      acc.x += w * v.x;
      acc.y += w * v.y;
      acc.z += w * v.z;
      acc.w += w * v.w;
      wsum += w;
    }
  }
  const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
  uint2 pk;
  pk.x = pack_bf16x2(acc.x * inv, acc.y * inv);
  pk.y = pack_bf16x2(acc.z * inv, acc.w * inv);
  *(uint2*)(p.out + ((int64_t)tok * H + h) * kValueDim + threadIdx.x * 4) = pk;
}

}  // namespace

cudaError_t launch_sfa(const SfaParams& p, cudaStream_t s) {
  cudaError_t e = cudaFuncSetAttribute(sfa_mma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       kSfaSmem);
  if (e != cudaSuccess) return e;
  dim3 grid(p.n_splits, (p.n_heads + kHB - 1) / kHB, p.tv.n_tokens);
  sfa_mma_kernel<<<grid, kSfaThreads, kSfaSmem, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_sfa_combine(const SfaParams& p, cudaStream_t s) {
  dim3 grid(p.n_heads, p.tv.n_tokens);
  sfa_combine_kernel<<<grid, 128, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace dsa
