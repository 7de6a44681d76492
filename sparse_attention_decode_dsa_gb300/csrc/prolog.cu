// Index prolog without weights: dynamic MXFP8 quantisation of index rows (queries or
// new keys) with groups of 32, optionally scattered into the paged K-index cache.
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
    const int b = a.tv.token_seq ? __ldg(a.tv.token_seq + row) : (int)row;
    if (b < 0 || b >= a.tv.batch) {
      if (part == 0) atomicOr(a.err, DSA_DEVERR_TOKEN);
      return;
    }
    const int pos = a.tv.token_pos ? __ldg(a.tv.token_pos + row) : __ldg(a.tv.seq_lens + b) - 1;
    if (pos < 0 || pos >= a.tv.max_pages * kPage) {
      if (part == 0) atomicOr(a.err, DSA_DEVERR_TOKEN);
      return;
    }
    const int page = __ldg(a.tv.block_table + (int64_t)b * a.tv.max_pages + (pos >> 6));
    if (page < 0 || page >= a.tv.num_pages) {
      if (part == 0) atomicOr(a.err, DSA_DEVERR_PAGE_ID);
      return;
    }
    dst = (int64_t)page * kPage + (pos & (kPage - 1));
  }

  const int e = amax > 0.f ? max(-127, min(127, floor_log2(amax) - 8)) : -127;
  const float mul = pow2(-e);
  uint2 out;
  out.x = cvt_e4m3x2(v[0] * mul, v[1] * mul) | (cvt_e4m3x2(v[2] * mul, v[3] * mul) << 16);
  out.y = cvt_e4m3x2(v[4] * mul, v[5] * mul) | (cvt_e4m3x2(v[6] * mul, v[7] * mul) << 16);
  *((uint2*)(a.codes + dst * a.dim) + part) = out;
  if ((part & 3) == 0) a.scales[dst * (a.dim >> 5) + (part >> 2)] = (uint8_t)(e + 127);
}

}  // namespace

cudaError_t launch_mxfp8_quant(const Mxfp8Params& p, cudaStream_t s) {
  const int64_t threads = p.n_rows * (p.dim >> 3);
  if (threads == 0) return cudaSuccess;
  const int64_t blocks = (threads + 255) / 256;
  mxfp8_quant_kernel<<<dim3((unsigned)blocks), dim3(256), 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace dsa
