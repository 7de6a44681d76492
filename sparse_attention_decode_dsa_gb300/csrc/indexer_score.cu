// Lightning Indexer, scoring pass: relevance scores, head weighting and head sum.
//
// "Adapting and Optimizing Inference for a New Model Architecture on Ascend", section
// 3.1: scores = query x paged keys^T, then weighted per head; the Top-K that follows
// keeps one score per key, so the weighted per-head scores are summed over heads.
// Keys are read straight from the paged cache ("Day0 Inference Optimization on Ascend
// CANN", section 2), with the MXFP8 group of 32 of section 3 for the quantised mode.
//
// Reference version on CUDA cores: one CTA per (query token, key page); thread
// (token s, lane j) accumulates the per-head dot products of heads j, j+4, ... in f32.
// With integer-valued inputs and power-of-two weights and scales every product and
// partial sum here is exact, so the result does not depend on the order of the sums.
#include "common.cuh"

namespace dsa {

namespace {

constexpr int kScoreThreads = 256;

template <int D, int KIND>  // KIND 0: bf16; 1: e4m3 + per-token f32; 2: e4m3 + E8M0/32
__global__ void __launch_bounds__(kScoreThreads) score_cuda_core_kernel(ScoreParams p) {
  constexpr int G = (KIND == 2) ? D / 32 : 1;  // scale groups per row
  const int row = blockIdx.y;
  const int pblk = blockIdx.x;
  pdl_trigger();
  pdl_wait();
  int b, n_vis;
  resolve_token(p.tv, row, &b, &n_vis, threadIdx.x == 0 ? p.err : nullptr);
  if (pblk * kPage >= n_vis) return;
  const int H = p.n_heads;

  __shared__ float qs[kMaxIdxHeads][D + 1];   // raw query values (scales kept apart)
  __shared__ float qgs[kMaxIdxHeads][G];      // query group scales (MX), else 1
  __shared__ float ws_[kMaxIdxHeads];         // head weights
  __shared__ float qtok_scale;

  for (int e = threadIdx.x; e < H * D; e += kScoreThreads) {
    int h = e / D, d = e % D;
    int64_t off = ((int64_t)row * H + h) * D + d;
    qs[h][d] = (KIND == 0) ? bf16_to_f32(((const uint16_t*)p.q)[off])
                           : e4m3_to_f32(((const uint8_t*)p.q)[off]);
  }
  for (int e = threadIdx.x; e < H * G; e += kScoreThreads) {
    int h = e / G, g = e % G;
    qgs[h][g] = (KIND == 2) ? e8m0_to_f32(((const uint8_t*)p.q_scale)[((int64_t)row * H + h) * G + g])
                            : 1.0f;
  }
  for (int h = threadIdx.x; h < H; h += kScoreThreads) ws_[h] = p.head_w[(int64_t)row * H + h];
  if (threadIdx.x == 0) qtok_scale = (KIND == 1) ? ((const float*)p.q_scale)[row] : 1.0f;
  __syncthreads();

  const int s = threadIdx.x >> 2;   // token slot in the page
  const int j = threadIdx.x & 3;    // head lane
  const int t = pblk * kPage + s;
  const bool valid = t < n_vis;
  int pg = physical_page(p.tv, b, pblk, (valid && j == 0 && s == 0) ? p.err : nullptr);

  float score = -INFINITY;
  if (valid && pg >= 0) {
    const int64_t krow = (int64_t)pg * kPage + s;
    float acc[kMaxIdxHeads / 4][G];
#pragma unroll
    for (int hh = 0; hh < kMaxIdxHeads / 4; ++hh)
#pragma unroll
      for (int g = 0; g < G; ++g) acc[hh][g] = 0.f;
    for (int d0 = 0; d0 < D; d0 += 8) {
      float kv[8];
      if (KIND == 0) {
        uint4 raw = *(const uint4*)((const uint16_t*)p.k + krow * D + d0);
        const uint16_t* r16 = (const uint16_t*)&raw;
#pragma unroll
        for (int u = 0; u < 8; ++u) kv[u] = bf16_to_f32(r16[u]);
      } else {
        uint2 raw = *(const uint2*)((const uint8_t*)p.k + krow * D + d0);
        const uint8_t* r8 = (const uint8_t*)&raw;
#pragma unroll
        for (int u = 0; u < 8; ++u) kv[u] = e4m3_to_f32(r8[u]);
      }
      const int g = (KIND == 2) ? d0 / 32 : 0;
#pragma unroll
      for (int hh = 0; hh < kMaxIdxHeads / 4; ++hh) {
        const int h = j + 4 * hh;
        if (h < H) {
          float a = 0.f;
#pragma unroll
          for (int u = 0; u < 8; ++u) a = fmaf(qs[h][d0 + u], kv[u], a);
#pragma unroll
          for (int gg = 0; gg < G; ++gg)
            if (gg == g) acc[hh][gg] += a;
        }
      }
    }
    float ksc[G];
    if (KIND == 1) {
      ksc[0] = ((const float*)p.k_scale)[krow];
    } else if (KIND == 2) {
#pragma unroll
      for (int g = 0; g < G; ++g) ksc[g] = e8m0_to_f32(((const uint8_t*)p.k_scale)[krow * G + g]);
    } else {
      ksc[0] = 1.f;
    }
    float part = 0.f;
#pragma unroll
    for (int hh = 0; hh < kMaxIdxHeads / 4; ++hh) {
      const int h = j + 4 * hh;
      if (h < H) {
        float hv = 0.f;  // this head's relevance score q_h . k_t, scales applied
#pragma unroll
        for (int g = 0; g < G; ++g) hv += acc[hh][g] * (ksc[g] * qgs[h][g]);
        hv *= qtok_scale;
        if (p.act == DSA_ACT_RELU) hv = fmaxf(hv, 0.f);
        hv *= ws_[h];      // head weighting
        part += hv;
      }
    }
    score = part;
  }
  // sum the four head lanes of this token
  score += __shfl_xor_sync(0xffffffffu, score, 1);
  score += __shfl_xor_sync(0xffffffffu, score, 2);
  if (valid && j == 0) {
    p.scores[(int64_t)row * p.score_stride + t] = score;
    atomicAdd(p.hist + (int64_t)row * kTopkBins + (score_key(score) >> 20), 1u);
  }
}

template <int D, int KIND>
cudaError_t launch_one(const ScoreParams& p, cudaStream_t s) {
  dim3 grid(p.max_page_blocks, p.tv.n_tokens);
  return launch_pdl(score_cuda_core_kernel<D, KIND>, grid, dim3(kScoreThreads), 0, s, p);
}

}  // namespace

cudaError_t launch_score(const ScoreParams& p, dsa_dtype_t dt, dsa_scale_t sk, cudaStream_t s) {
  const int kind = (dt == DSA_BF16) ? 0 : (sk == DSA_SCALE_PER_TOKEN_F32 ? 1 : 2);
  if (p.dim == 64) {
    if (kind == 0) return launch_one<64, 0>(p, s);
    if (kind == 1) return launch_one<64, 1>(p, s);
    return launch_one<64, 2>(p, s);
  }
  if (kind == 0) return launch_one<128, 0>(p, s);
  if (kind == 1) return launch_one<128, 1>(p, s);
  return launch_one<128, 2>(p, s);
}

}  // namespace dsa
