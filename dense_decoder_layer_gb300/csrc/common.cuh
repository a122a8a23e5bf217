// Device helpers shared by the kernels of the dense prefill stack.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace pds {

// Bits of the plan's device status word.
enum : uint32_t {
  kStatusTimeout = 1u,      // a bounded mbarrier / flag wait gave up
  kStatusBadSchedule = 2u,  // a kernel met a work split it cannot serve
};

__device__ __forceinline__ float bf16_to_f32(uint16_t b) { return __uint_as_float(uint32_t(b) << 16); }

__device__ __forceinline__ uint16_t f32_to_bf16(float f) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}

// Two float32 as bf16 (round to nearest even) in one 32-bit word, lo in
// the low half: one paired conversion.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

__device__ __forceinline__ float silu(float t) { return __fdividef(t, 1.0f + __expf(-t)); }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Row scale of RMSNorm from the row's sum-of-squares partials (one per
// 64-column group of the row, written by the producing epilogue).
__device__ __forceinline__ float rms_row_scale(const float* ss_row, int nparts, float inv_d,
                                               float eps) {
  float t = 0.f;
  for (int i = 0; i < nparts; ++i) t += ss_row[i];
  return rsqrtf(t * inv_d + eps);
}

}  // namespace pds
