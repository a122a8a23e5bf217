// Once-per-call kernels of the dense prefill stack: the RoPE table of the
// call's positions and the first layer's norm prep.  Both are small and
// bound by memory or latency; everything else of a layer runs inside the
// tensor-core kernels' epilogues.
#include <math.h>

#include "common.cuh"
#include "kernels.h"

namespace pds {
namespace {

// (c, s) = mscale * (cos, sin)(p * omega_i) for pair i and row b, p = start_pos
// + b.  The angle is formed and reduced to [-pi, pi] in float64 (positions
// reach tens of thousands of radians, where a float32 angle would be off by
// milliradians), then the reduced angle's sine and cosine are taken in
// float32.
__global__ void rope_table_kernel(float2* __restrict__ table, int M, int start_pos, RopeFreqs f) {
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= M * f.n_pairs) return;
  const int i = t / M, b = t - (t / M) * M;  // table laid out [pair][row]
  constexpr double kTwoPi = 6.283185307179586476925286766559;
  const double ang = static_cast<double>(start_pos + b) * f.omega[i];
  const double red = ang - rint(ang / kTwoPi) * kTwoPi;
  float s, c;
  sincosf(static_cast<float>(red), &s, &c);
  table[t] = make_float2(c * f.mscale, s * f.mscale);
}

// a = bf16(x * gain) and the sum of squares of x per 64-column group of a
// row.  One warp per 128 columns of a row: lanes 0-15 hold group 2k, lanes
// 16-31 group 2k+1, four columns per lane (16-byte loads).
__global__ void __launch_bounds__(256) norm_prep_kernel(const float* __restrict__ x,
                                                        const float* __restrict__ gain,
                                                        uint16_t* __restrict__ a_out,
                                                        float* __restrict__ ss_out, int M, int d) {
  const int units_per_row = d / 128;
  const int unit = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (unit >= M * units_per_row) return;
  const int b = unit / units_per_row, c0 = (unit - b * units_per_row) * 128;
  const size_t off = static_cast<size_t>(b) * d + c0 + 4 * lane;
  const float4 v = __ldcs(reinterpret_cast<const float4*>(x + off));
  const float4 g = __ldg(reinterpret_cast<const float4*>(gain + c0) + lane);
  *reinterpret_cast<uint2*>(a_out + off) =
      make_uint2(pack_bf16x2(v.x * g.x, v.y * g.y), pack_bf16x2(v.z * g.z, v.w * g.w));
  float s = __fadd_rn(__fadd_rn(__fmul_rn(v.x, v.x), __fmul_rn(v.y, v.y)),
                      __fadd_rn(__fmul_rn(v.z, v.z), __fmul_rn(v.w, v.w)));
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  if ((lane & 15) == 0) ss_out[static_cast<size_t>(b) * (d / 64) + c0 / 64 + (lane >> 4)] = s;
}

}  // namespace

void launch_rope_table(float2* table, int M, int start_pos, const RopeFreqs& f, cudaStream_t st) {
  const int n = M * f.n_pairs;
  if (n > 0) rope_table_kernel<<<(n + 255) / 256, 256, 0, st>>>(table, M, start_pos, f);
}

void launch_norm_prep(const float* x, const float* gain, uint16_t* a_out, float* ss_out, int M,
                      int d, cudaStream_t st) {
  const int units = M * (d / 128);
  norm_prep_kernel<<<(units + 7) / 8, 256, 0, st>>>(x, gain, a_out, ss_out, M, d);
}

}  // namespace pds
