// Straightforward SIMT kernels of every step of the dense prefill stack.
//
// They are the stack's first, unfused CUDA path: a float32-accumulating
// GEMM into a float32 scratch matrix followed by one elementwise epilogue
// kernel per fused epilogue of the tensor-core path, and an attention
// kernel with one CTA per (query row, head).  They compute the same
// function with the same roundings (bf16 operands and outputs, float32
// everywhere else) and serve as the cross-check of the fast kernels.
#include "common.cuh"
#include "kernels.h"

namespace pds {
namespace {

constexpr int kTile = 64;
constexpr int kTk = 32;

__global__ void __launch_bounds__(256) gemm_naive_kernel(const uint16_t* __restrict__ A,
                                                         WeightRows W, float* __restrict__ C,
                                                         int M, int N, int K) {
  __shared__ float As[kTk][kTile + 1];
  __shared__ float Ws[kTk][kTile + 1];
  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
  const int m0 = blockIdx.y * kTile, n0 = blockIdx.x * kTile;
  float acc[4][4] = {};
  for (int k0 = 0; k0 < K; k0 += kTk) {
    for (int i = threadIdx.x; i < kTile * kTk; i += 256) {
      int r = i / kTk, c = i % kTk;
      int m = m0 + r, n = n0 + r, k = k0 + c;
      As[c][r] = (m < M && k < K) ? bf16_to_f32(A[(size_t)m * K + k]) : 0.f;
      float wv = 0.f;
      if (n < N && k < K) {
        int blk = 0, row = n;
        while (blk < W.n - 1 && row >= W.rows[blk]) row -= W.rows[blk++];
        wv = bf16_to_f32(W.w[blk][(size_t)row * K + k]);
      }
      Ws[c][r] = wv;
    }
    __syncthreads();
#pragma unroll 8
    for (int c = 0; c < kTk; ++c) {
      float a[4], w[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[c][ty + 16 * i];
#pragma unroll
      for (int j = 0; j < 4; ++j) w[j] = Ws[c][tx + 16 * j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], w[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      int m = m0 + ty + 16 * i, n = n0 + tx + 16 * j;
      if (m < M && n < N) C[(size_t)m * N + n] = acc[i][j];
    }
}

// One CTA per row.
__global__ void qkv_epilogue_kernel(const float* __restrict__ C, QkvEpilogue e) {
  const int b = blockIdx.x;
  const int N = e.q_width + 2 * e.kv_width;
  const int half = e.head_dim / 2;
  const float r = rms_row_scale(e.rs.ss + (size_t)b * e.rs.ss_parts, e.rs.ss_parts, e.rs.inv_d,
                                e.rs.eps);
  const float* row = C + (size_t)b * N;
  // q and k: rotate the pairs (i, i + hd/2) of every head
  const int n_rot_heads = (e.q_width + e.kv_width) / e.head_dim;
  for (int t = threadIdx.x; t < n_rot_heads * half; t += blockDim.x) {
    const int hh = t / half, i = t % half;
    const int c0 = hh * e.head_dim + i;
    const float u = r * row[c0], w = r * row[c0 + half];
    const float2 sc = e.rope[(size_t)i * e.rope_ld + b];
    const float o0 = u * sc.x - w * sc.y, o1 = u * sc.y + w * sc.x;
    uint16_t* dst;
    if (c0 < e.q_width) {
      dst = e.q + (size_t)b * e.q_width + c0;
    } else {
      dst = e.k_cache + (size_t)(e.start_pos + b) * e.kv_width + (c0 - e.q_width);
    }
    dst[0] = f32_to_bf16(o0);
    dst[half] = f32_to_bf16(o1);
  }
  for (int c = threadIdx.x; c < e.kv_width; c += blockDim.x) {
    e.v_cache[(size_t)(e.start_pos + b) * e.kv_width + c] =
        f32_to_bf16(r * row[e.q_width + e.kv_width + c]);
  }
}

// One CTA (8 warps) per row; a warp per 64-column group of the statistics.
__global__ void resid_epilogue_kernel(const float* __restrict__ C, ResidEpilogue e, int N) {
  const int b = blockIdx.x;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int groups = N / 64;
  for (int gi = warp; gi < groups; gi += blockDim.x / 32) {
    float ss = 0.f;
    for (int j = lane; j < 64; j += 32) {
      const size_t idx = (size_t)b * N + gi * 64 + j;
      float hv = e.resid[idx] + (C ? C[idx] : 0.f);
      if (e.out) e.out[idx] = hv;
      if (e.gain) {
        e.a_out[idx] = f32_to_bf16(hv * e.gain[gi * 64 + j]);
        ss += hv * hv;
      }
    }
    ss = warp_sum(ss);
    if (e.gain && lane == 0) e.ss_out[(size_t)b * groups + gi] = ss;
  }
}

__global__ void swiglu_epilogue_kernel(const float* __restrict__ C, SwigluEpilogue e) {
  const int b = blockIdx.x;
  const float r = rms_row_scale(e.rs.ss + (size_t)b * e.rs.ss_parts, e.rs.ss_parts, e.rs.inv_d,
                                e.rs.eps);
  const float* row = C + (size_t)b * 2 * e.ffn;
  for (int f = threadIdx.x; f < e.ffn; f += blockDim.x) {
    const float g = r * row[f], u = r * row[e.ffn + f];
    e.act[(size_t)b * e.ffn + f] = f32_to_bf16(silu(g) * u);
  }
}

// One CTA per (row b, head h): scores of all visible keys in shared memory.
__global__ void attention_naive_kernel(const uint16_t* __restrict__ q,
                                       const uint16_t* __restrict__ k,
                                       const uint16_t* __restrict__ v, uint16_t* __restrict__ o,
                                       int start_pos, int H, int Hkv, int hd) {
  extern __shared__ float smem[];
  float* qs = smem;        // [hd]
  float* sc = smem + hd;   // [T]
  __shared__ float red[32];
  const int b = blockIdx.x, h = blockIdx.y;
  const int g = h / (H / Hkv);
  const int T = start_pos + b + 1;
  const float scale = rsqrtf((float)hd);
  for (int c = threadIdx.x; c < hd; c += blockDim.x)
    qs[c] = bf16_to_f32(q[((size_t)b * H + h) * hd + c]);
  __syncthreads();
  float mx = -INFINITY;
  for (int j = threadIdx.x; j < T; j += blockDim.x) {
    const uint16_t* kr = k + ((size_t)j * Hkv + g) * hd;
    float s = 0.f;
    for (int c = 0; c < hd; ++c) s = fmaf(qs[c], bf16_to_f32(kr[c]), s);
    s *= scale;
    sc[j] = s;
    mx = fmaxf(mx, s);
  }
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32, nw = blockDim.x / 32;
  mx = warp_max(mx);
  if (lane == 0) red[warp] = mx;
  __syncthreads();
  mx = red[0];
  for (int i = 1; i < nw; ++i) mx = fmaxf(mx, red[i]);
  __syncthreads();
  float sum = 0.f;
  for (int j = threadIdx.x; j < T; j += blockDim.x) {
    const float p = __expf(sc[j] - mx);
    sc[j] = p;
    sum += p;
  }
  sum = warp_sum(sum);
  if (lane == 0) red[warp] = sum;
  __syncthreads();
  sum = 0.f;
  for (int i = 0; i < nw; ++i) sum += red[i];
  const float inv = 1.f / sum;
  for (int c = threadIdx.x; c < hd; c += blockDim.x) {
    float acc = 0.f;
    for (int j = 0; j < T; ++j) acc = fmaf(sc[j], bf16_to_f32(v[((size_t)j * Hkv + g) * hd + c]), acc);
    o[(size_t)b * H * hd + h * hd + c] = f32_to_bf16(acc * inv);
  }
}

__global__ void rope_table_kernel(float2* table, int M, int start_pos, int half, double theta,
                                  int head_dim) {
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= M * half) return;
  const int i = t / M, b = t % M;  // table laid out [channel][row]
  const double omega = pow(theta, -2.0 * i / head_dim);
  double s, c;
  sincos((double)(start_pos + b) * omega, &s, &c);
  table[t] = make_float2((float)c, (float)s);
}

}  // namespace

void launch_rope_table(float2* table, int M, int start_pos, int half, double theta, int head_dim,
                       cudaStream_t st) {
  const int n = M * half;
  rope_table_kernel<<<(n + 255) / 256, 256, 0, st>>>(table, M, start_pos, half, theta, head_dim);
}

void launch_norm_prep(const float* x, const float* gain, uint16_t* a_out, float* ss_out, int M,
                      int d, cudaStream_t st) {
  ResidEpilogue e{x, nullptr, gain, a_out, ss_out};
  resid_epilogue_kernel<<<M, 256, 0, st>>>(nullptr, e, d);
}

void launch_gemm_naive(const uint16_t* A, const WeightRows& W, float* C, int M, int N, int K,
                       cudaStream_t st) {
  dim3 grid((N + kTile - 1) / kTile, (M + kTile - 1) / kTile);
  gemm_naive_kernel<<<grid, 256, 0, st>>>(A, W, C, M, N, K);
}

void launch_qkv_epilogue_naive(const float* C, const QkvEpilogue& e, int M, cudaStream_t st) {
  qkv_epilogue_kernel<<<M, 256, 0, st>>>(C, e);
}

void launch_resid_epilogue_naive(const float* C, const ResidEpilogue& e, int M, int N,
                                 cudaStream_t st) {
  resid_epilogue_kernel<<<M, 256, 0, st>>>(C, e, N);
}

void launch_swiglu_epilogue_naive(const float* C, const SwigluEpilogue& e, int M,
                                  cudaStream_t st) {
  swiglu_epilogue_kernel<<<M, 256, 0, st>>>(C, e);
}

void launch_attention_naive(const uint16_t* q, const uint16_t* k, const uint16_t* v, uint16_t* o,
                            int B, int start_pos, int H, int Hkv, int hd, cudaStream_t st) {
  const int T = start_pos + B;
  const size_t smem = sizeof(float) * (hd + T);
  if (smem > 48 * 1024)
    cudaFuncSetAttribute(attention_naive_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         (int)smem);
  attention_naive_kernel<<<dim3(B, H), 128, smem, st>>>(q, k, v, o, start_pos, H, Hkv, hd);
}

}  // namespace pds
