// Prolog without weights: dynamic MXFP8 quantisation of index rows (queries or new keys)
// with groups of 32, optionally scattered into the paged K-index cache; and the append of
// each new token's key to a bf16 or per-token-FP8 K-index cache and of its latent row to
// a bf16 or FP8 (tiles of 128) latent cache.
//
// MXFP8 with per-group dynamic quantisation and a group of 32 elements is the index
// path's format ("Day0 Inference Optimization on Ascend CANN", section 3, "Full
// Quantization of LI with MXFP8"; "Adapting and Optimizing Inference for a New Model
// Architecture on Ascend", section 4.2).  The pages leave the scale rule open; this
// follows the OCP microscaling one: a group's shared exponent is
// e = floor(log2(amax)) - 8 (8: the exponent of E4M3's largest normal, 448), clamped to
// [-127, 127] (-127 for an all-zero group), stored as the E8M0 byte e + 127, and each
// element is x * 2^-e rounded to the nearest E4M3 value (ties to even), saturating at
// 448.  x * 2^-e is exact in f32 wherever the rounding can tell values apart, so the
// codes are those of the exact quotient.
//
// HBM-bound elementwise work: each thread takes 8 consecutive bf16 (one 16-byte load)
// and writes 8 codes (8 bytes); the four threads of a 32-element group meet through two
// shuffles for the group maximum, and the first of them writes the scale byte.
#include "common.cuh"
#include "dsa_internal.h"

namespace dsa {
namespace {

// floor(log2(a)) for a finite f32 a > 0 (normal or subnormal), from its bits.
__device__ __forceinline__ int floor_log2(float a) {
  const uint32_t u = __float_as_uint(a);
  const int ex = (int)(u >> 23);
  if (ex > 0) return ex - 127;
  return (31 - __clz((int)(u & 0x7FFFFFu))) - 149;
}

// 2^s as an f32 for s in [-127, 127] (2^-127 is subnormal).
__device__ __forceinline__ float pow2(int s) {
  return s >= -126 ? __uint_as_float((uint32_t)(s + 127) << 23) : __uint_as_float(0x00400000u);
}

// Two f32 -> two E4M3 codes (round to nearest even, saturating), `lo` in the low byte.
__device__ __forceinline__ uint32_t cvt_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;\n" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Cache row (page * 64 + slot) of the new row of token `row`, or -1 (with an error bit,
// reported by the thread with `lead`) when its position or page is outside the table:
// batch row token_seq[row] (or row), position token_pos[row] (or seq_len - 1).
__device__ __forceinline__ int64_t append_dst(const TokenView& tv, int64_t row, uint32_t* err, bool lead) {
  const int b = tv.token_seq ? __ldg(tv.token_seq + row) : (int)row;
  if (b < 0 || b >= tv.batch) {
    if (lead) atomicOr(err, DSA_DEVERR_TOKEN);
    return -1;
  }
  const int pos = tv.token_pos ? __ldg(tv.token_pos + row) : __ldg(tv.seq_lens + b) - 1;
  if (pos < 0 || pos >= tv.max_pages * kPage) {
    if (lead) atomicOr(err, DSA_DEVERR_TOKEN);
    return -1;
  }
  const int page = __ldg(tv.block_table + (int64_t)b * tv.max_pages + (pos >> 6));
  if (page < 0 || page >= tv.num_pages) {
    if (lead) atomicOr(err, DSA_DEVERR_PAGE_ID);
    return -1;
  }
  return (int64_t)page * kPage + (pos & (kPage - 1));
}

__global__ void __launch_bounds__(256) mxfp8_quant_kernel(Mxfp8Params a) {
  const int per_row = a.dim >> 3;  // threads per row; a multiple of 4 (dim % 32 == 0)
  const int64_t gid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const bool valid = gid < a.n_rows * per_row;
  const int64_t row = valid ? gid / per_row : 0;
  const int part = valid ? (int)(gid - row * per_row) : 0;
  uint4 raw = make_uint4(0u, 0u, 0u, 0u);
  if (valid) raw = __ldg((const uint4*)(a.x + row * a.dim) + part);
  const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
  float v[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[2 * i] = __uint_as_float(w[i] << 16);
    v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(v[i]));
  // a group's four threads are consecutive lanes (rows start on multiples of 4 threads);
  // every lane takes part, in range or not
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
  if (!valid) return;

  int64_t dst = row;
  if (a.append) {  // the new key of token `row` goes to its (page, slot)
    dst = append_dst(a.tv, row, a.err, part == 0);
    if (dst < 0) return;
  }

  const int e = amax > 0.f ? max(-127, min(127, floor_log2(amax) - 8)) : -127;
  const float mul = pow2(-e);
  uint2 out;
  out.x = cvt_e4m3x2(v[0] * mul, v[1] * mul) | (cvt_e4m3x2(v[2] * mul, v[3] * mul) << 16);
  out.y = cvt_e4m3x2(v[4] * mul, v[5] * mul) | (cvt_e4m3x2(v[6] * mul, v[7] * mul) << 16);
  *((uint2*)(a.codes + dst * a.dim) + part) = out;
  if ((part & 3) == 0) a.scales[dst * (a.dim >> 5) + (part >> 2)] = (uint8_t)(e + 127);
}

// FP8 block quantisation (absmax): the block's f32 scale is amax / 448 (1 for an
// all-zero block), each element the E4M3 value nearest to x / scale (ties to even,
// saturating).  Both divisions are IEEE binary32 divisions (__fdiv_rn), so the codes
// are those of the correctly rounded quotient.
__device__ __forceinline__ float fp8_block_scale(float amax) { return amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f; }

// The new latent row of each token appended to the paged latent cache.  One CTA of 128
// threads per token.  bf16 cache: the 1152-byte row copied (72 x 16 B).  FP8 cache: warp
// w quantises latent tile w (dims 128 w .. 128 w + 127, 4 per lane, the tile maximum
// through five shuffles) into codes [.., 512] and scale [.., 4]; 8 threads copy the 64
// rope dims (bf16) to rope [.., 64].
template <bool FP8>
__global__ void __launch_bounds__(128) latent_append_kernel(LatentAppendParams a) {
  const int64_t row = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int64_t dst = append_dst(a.tv, row, a.err, tid == 0);
  if (dst < 0) return;  // (uniform over the CTA)
  const uint16_t* x = a.x + row * kLatentDim;
  if (!FP8) {
    if (tid < kLatentDim / 8)
      *((uint4*)(a.data + dst * kLatentDim) + tid) = __ldg((const uint4*)x + tid);
    return;
  }
  const uint2 raw = __ldg((const uint2*)(x + 128 * w) + lane);
  const float v[4] = {__uint_as_float(raw.x << 16), __uint_as_float(raw.x & 0xFFFF0000u),
                      __uint_as_float(raw.y << 16), __uint_as_float(raw.y & 0xFFFF0000u)};
  float amax = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
#pragma unroll
  for (int o = 16; o; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const float sc = fp8_block_scale(amax);
  const uint32_t codes = cvt_e4m3x2(__fdiv_rn(v[0], sc), __fdiv_rn(v[1], sc)) |
                         (cvt_e4m3x2(__fdiv_rn(v[2], sc), __fdiv_rn(v[3], sc)) << 16);
  *((uint32_t*)(a.codes + dst * kValueDim + 128 * w) + lane) = codes;
  if (lane == 0) a.scales[dst * (kValueDim / 128) + w] = sc;
  if (tid < (kLatentDim - kValueDim) / 8)
    *((uint4*)(a.rope + dst * (kLatentDim - kValueDim)) + tid) = __ldg((const uint4*)(x + kValueDim) + tid);
}

// New keys appended to a bf16 K-index cache (copied) or an e4m3 one with one f32 scale
// per token (FP8 block quantisation of the whole row).  One warp per token, D / 32
// elements per lane.
template <int D, bool FP8>
__global__ void __launch_bounds__(128) index_append_kernel(IndexAppendParams a) {
  const int64_t row = (int64_t)blockIdx.x * 4 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= a.n_rows) return;
  const int64_t dst = append_dst(a.tv, row, a.err, lane == 0);
  if (dst < 0) return;  // (uniform over the warp)
  constexpr int E = D / 32;  // elements per lane: 2 or 4
  const uint16_t* x = a.x + row * D + E * lane;
  if (!FP8) {
    if (E == 4) *((uint2*)((uint16_t*)a.data + dst * D) + lane) = __ldg((const uint2*)x);
    else *((uint32_t*)((uint16_t*)a.data + dst * D) + lane) = __ldg((const uint32_t*)x);
    return;
  }
  float v[4] = {0.f, 0.f, 0.f, 0.f};
  if (E == 4) {
    const uint2 raw = __ldg((const uint2*)x);
    v[0] = __uint_as_float(raw.x << 16);
    v[1] = __uint_as_float(raw.x & 0xFFFF0000u);
    v[2] = __uint_as_float(raw.y << 16);
    v[3] = __uint_as_float(raw.y & 0xFFFF0000u);
  } else {
    const uint32_t raw = __ldg((const uint32_t*)x);
    v[0] = __uint_as_float(raw << 16);
    v[1] = __uint_as_float(raw & 0xFFFF0000u);
  }
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < E; ++i) amax = fmaxf(amax, fabsf(v[i]));
#pragma unroll
  for (int o = 16; o; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const float sc = fp8_block_scale(amax);
  uint8_t* cdst = (uint8_t*)a.data + dst * D + E * lane;
  const uint32_t c01 = cvt_e4m3x2(__fdiv_rn(v[0], sc), __fdiv_rn(v[1], sc));
  if (E == 4) *(uint32_t*)cdst = c01 | (cvt_e4m3x2(__fdiv_rn(v[2], sc), __fdiv_rn(v[3], sc)) << 16);
  else *(uint16_t*)cdst = (uint16_t)c01;
  if (lane == 0) a.scales[dst] = sc;
}

}  // namespace

cudaError_t launch_latent_append(const LatentAppendParams& p, bool fp8, cudaStream_t s) {
  if (p.n_rows == 0) return cudaSuccess;
  if (fp8) latent_append_kernel<true><<<dim3((unsigned)p.n_rows), dim3(128), 0, s>>>(p);
  else latent_append_kernel<false><<<dim3((unsigned)p.n_rows), dim3(128), 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_index_append(const IndexAppendParams& p, int dim, bool fp8, cudaStream_t s) {
  if (p.n_rows == 0) return cudaSuccess;
  const dim3 g((unsigned)((p.n_rows + 3) / 4)), t(128);
  if (dim == 64) {
    if (fp8) index_append_kernel<64, true><<<g, t, 0, s>>>(p);
    else index_append_kernel<64, false><<<g, t, 0, s>>>(p);
  } else {
    if (fp8) index_append_kernel<128, true><<<g, t, 0, s>>>(p);
    else index_append_kernel<128, false><<<g, t, 0, s>>>(p);
  }
  return cudaGetLastError();
}

cudaError_t launch_mxfp8_quant(const Mxfp8Params& p, cudaStream_t s) {
  const int64_t threads = p.n_rows * (p.dim >> 3);
  if (threads == 0) return cudaSuccess;
  const int64_t blocks = (threads + 255) / 256;
  mxfp8_quant_kernel<<<dim3((unsigned)blocks), dim3(256), 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace dsa
