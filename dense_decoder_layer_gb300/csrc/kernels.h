// Internal launch interface between the host library and the kernel files.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace pds {

// A weight operand made of up to three row blocks [rows_i, K] stacked
// along N (wq|wk|wv for the fused QKV projection, gate|up for the FFN).
struct WeightRows {
  const uint16_t* w[3];
  int rows[3];
  int n;  // number of blocks in use
};

// ---- epilogue descriptions (shared by the naive and tensor-core paths) ----

// RMSNorm row scale from sum-of-squares partials [M, ss_parts], one per
// 64-column group of the row.
struct RowScale {
  const float* ss;  // [M, ss_parts]
  int ss_parts;
  float inv_d;
  float eps;
};

// QKV epilogue: scale rows, rotate q and k (NeoX half layout, table
// [M, hd/2] of (cos, sin) at each row's position), write q and the new
// cache rows.
struct QkvEpilogue {
  RowScale rs;
  const float2* rope;  // [hd/2, rope_ld]: channel i of row b at rope[i * rope_ld + b]
  int rope_ld;         // row stride of the table (the batch size)
  uint16_t* q;         // [M, H*hd]
  uint16_t* k_cache;   // [cap, Hkv*hd]; row b goes to row start_pos+b
  uint16_t* v_cache;
  int start_pos;
  int q_width, kv_width, head_dim;
};

// Residual epilogue: out = resid + acc (float32), and for a following
// norm: a = bf16(out * gain) and per-64-column sum-of-squares partials.
struct ResidEpilogue {
  const float* resid;  // [M, N]
  float* out;          // [M, N]
  const float* gain;   // [N] or nullptr (no following norm)
  uint16_t* a_out;     // [M, N] bf16
  float* ss_out;       // [M, N/64]
};

// SwiGLU epilogue: act = silu(r*gate) * (r*up), bf16 [M, F].
struct SwigluEpilogue {
  RowScale rs;
  uint16_t* act;  // [M, F]
  int ffn;
};

// ---------------------------------------------------------------- launches

// (cos, sin) of pos*omega_i for pos = start_pos + b, b < M, i < hd/2, laid
// out [i][b] (table[i * M + b]).
void launch_rope_table(float2* table, int M, int start_pos, int half, double theta,
                       int head_dim, cudaStream_t st);

// First-layer norm prep: a = bf16(x * gain), ss partials.
void launch_norm_prep(const float* x, const float* gain, uint16_t* a_out, float* ss_out, int M,
                      int d, cudaStream_t st);

// Naive (SIMT) path: C = A . W^T into float32, then separate epilogues.
void launch_gemm_naive(const uint16_t* A, const WeightRows& W, float* C, int M, int N, int K,
                       cudaStream_t st);
void launch_qkv_epilogue_naive(const float* C, const QkvEpilogue& e, int M, cudaStream_t st);
void launch_resid_epilogue_naive(const float* C, const ResidEpilogue& e, int M, int N,
                                 cudaStream_t st);
void launch_swiglu_epilogue_naive(const float* C, const SwigluEpilogue& e, int M,
                                  cudaStream_t st);
void launch_attention_naive(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                            uint16_t* o, int B, int start_pos, int H, int Hkv, int hd,
                            cudaStream_t st);

}  // namespace pds
