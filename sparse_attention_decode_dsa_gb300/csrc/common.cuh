// Device helpers shared by the kernels: token resolution, number formats, async copies,
// warp-level matrix fragments.
#pragma once
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "dsa_internal.h"

namespace dsa {

// ---- query-token resolution --------------------------------------------------------
// Batch row of token i and the number of positions it may select (t <= pos, t < len).
// Out-of-range metadata sets an error bit and yields an empty visible range.
__device__ __forceinline__ void resolve_token(const TokenView& tv, int i, int* b_out,
                                              int* n_out, uint32_t* err) {
  int b = tv.token_seq ? __ldg(tv.token_seq + i) : i;
  if (b < 0 || b >= tv.batch) {
    if (err) atomicOr(err, DSA_DEVERR_TOKEN);
    *b_out = 0;
    *n_out = 0;
    return;
  }
  int len = __ldg(tv.seq_lens + b);
  if (len < 0 || len > tv.max_pages * kPage) {
    if (err) atomicOr(err, DSA_DEVERR_SEQ_LEN);
    len = len < 0 ? 0 : tv.max_pages * kPage;
  }
  int pos = tv.token_pos ? __ldg(tv.token_pos + i) : len - 1;
  if (pos < -1) {
    if (err) atomicOr(err, DSA_DEVERR_TOKEN);
    pos = -1;
  }
  int n = pos + 1 < len ? pos + 1 : len;
  if (n > tv.max_visible) {  // device metadata disagrees with the host copy used to plan
    if (err) atomicOr(err, DSA_DEVERR_SEQ_LEN);
    n = tv.max_visible;
  }
  *b_out = b;
  *n_out = n;
}

// Physical page of logical page j of batch row b, or -1 (with an error bit) if the
// table entry is outside the cache.
__device__ __forceinline__ int physical_page(const TokenView& tv, int b, int j, uint32_t* err) {
  int pg = __ldg(tv.block_table + (int64_t)b * tv.max_pages + j);
  if (pg < 0 || pg >= tv.num_pages) {
    if (err) atomicOr(err, DSA_DEVERR_PAGE_ID);
    return -1;
  }
  return pg;
}

// ---- number formats -----------------------------------------------------------------
__device__ __forceinline__ float bf16_to_f32(uint16_t h) { return __uint_as_float((uint32_t)h << 16); }

__device__ __forceinline__ float e4m3_to_f32(uint8_t v) {
  __half_raw hr = __nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)v, __NV_E4M3);
  return __half2float(__half(hr));
}

// E8M0 exponent byte -> 2^(e-127) as f32 (e = 0 gives the subnormal 2^-127, 0xFF NaN).
// Branch-free (selects), so that loops over loaded bytes keep their loads in flight.
__device__ __forceinline__ float e8m0_to_f32(uint8_t e) {
  const uint32_t u = e == 0 ? 0x00400000u : (e == 0xFF ? 0x7FC00000u : (uint32_t)e << 23);
  return __uint_as_float(u);
}

// f32 -> bf16 bits, round to nearest even (NaN kept quiet).
__device__ __forceinline__ uint16_t f32_to_bf16_rne(float f) {
  uint32_t u = __float_as_uint(f);
  if ((u & 0x7FFFFFFFu) > 0x7F800000u) return (uint16_t)((u >> 16) | 0x40);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  return (uint32_t)f32_to_bf16_rne(lo) | ((uint32_t)f32_to_bf16_rne(hi) << 16);
}

// Order-preserving unsigned key of a float: larger score <-> larger key; -0 == +0.
__device__ __forceinline__ uint32_t score_key(float f) {
  uint32_t u = __float_as_uint(f);
  if ((u << 1) == 0u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_score(uint32_t k) {
  uint32_t u = (k & 0x80000000u) ? (k ^ 0x80000000u) : ~k;
  return __uint_as_float(u);
}

// ---- async copies and warp matrix fragments ---------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

// Programmatic dependent launch.  pdl_trigger: this CTA no longer holds back the launch
// of the next kernel in the stream (which may then start its own set-up early);
// pdl_wait: wait until the previous kernel in the stream has completed and its memory
// writes are visible.  Both are no-ops for a kernel launched without the attribute.
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }

// 16-byte read-only load that bypasses L1 allocation (streamed once).
__device__ __forceinline__ uint4 ldg_nc_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];\n"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

}  // namespace dsa
