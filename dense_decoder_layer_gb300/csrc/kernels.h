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

// ---- epilogue descriptions of the tensor-core GEMMs ----

// RMSNorm row scale from sum-of-squares partials [M, ss_parts], one per
// 64-column group of the row.
struct RowScale {
  const float* ss;  // [M, ss_parts]
  int ss_parts;
  float inv_d;
  float eps;
};

// QKV epilogue: scale rows, add the biases, RMSNorm every q / k head with
// its gain, rotate q and k (table [rot_dim/2, M] of (cos, sin) * mscale at
// each row's position), write q and the new cache rows.
struct QkvEpilogue {
  RowScale rs;
  const float2* rope;  // [rot_dim/2, rope_ld]: pair i of row b at rope[i * rope_ld + b]
  int rope_ld;         // row stride of the table (the batch size)
  uint16_t* q;         // [M, H*hd]
  uint16_t* k_cache;   // [cap, Hkv*hd]; row b goes to row start_pos+b
  uint16_t* v_cache;
  int start_pos;
  int q_width, kv_width, head_dim;
  // Variants (the general epilogue; the fast one serves Neox over the whole
  // head with no extras).
  int rope_layout;         // PDS_ROPE_NEOX / PDS_ROPE_NORM
  int rot_dim;             // rotated channels per head
  const float* bias[3];    // q [H*hd], k [Hkv*hd], v [Hkv*hd]; each may be null
  const float* norm[2];    // q, k head norm gains [hd]; each may be null
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

// Angular frequencies of the rotated pairs and the scale of the rotated
// channels: pair i of a head turns by p * omega[i] at position p, and
// cos/sin are multiplied by mscale.  omega is formed on the host in
// float64.
constexpr int kMaxRopePairs = 64;
struct RopeFreqs {
  double omega[kMaxRopePairs];
  int n_pairs;  // rot_dim / 2
  float mscale;
};

// (cos, sin) * mscale of p*omega_i for p = start_pos + b, b < M, i < n_pairs,
// laid out [i][b] (table[i * M + b]).
void launch_rope_table(float2* table, int M, int start_pos, const RopeFreqs& f, cudaStream_t st);

// First-layer norm prep: a = bf16(x * gain), ss partials [M, d/64].
void launch_norm_prep(const float* x, const float* gain, uint16_t* a_out, float* ss_out, int M,
                      int d, cudaStream_t st);

}  // namespace pds
