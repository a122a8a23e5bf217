// Tensor-core (tcgen05 / TMA) kernels of the stack: launch interface.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <string>

#include "../../include/pds.h"
#include "kernels.h"

namespace pds {

struct TmapCache;  // tensor maps already encoded, keyed by (pointer, shape)

struct TcContext {
  int num_sms = 0;
  uint32_t* status = nullptr;  // device status word (bounded waits)
  char* ws = nullptr;          // GEMM scratch: stream-K partial tiles, tile counters
  size_t ws_bytes = 0;
  char* attn_ws = nullptr;     // attention scratch: partial rows of chunked key ranges
  size_t attn_ws_bytes = 0;    // 0: no chunked mode
  TmapCache* maps = nullptr;   // optional
  bool pdl = false;            // launch with programmatic stream serialization
};

// Largest grid of the persistent GEMM (partial-tile scratch is sized by it).
constexpr int kGemmMaxGrid = 192;

// Scratch bytes the tensor-core GEMMs need for an M-row problem whose
// largest GEMM has `max_tiles_n` column tiles.
size_t tc_gemm_scratch_bytes(int M, int max_tiles_n);

TmapCache* tmap_cache_create();
void tmap_cache_destroy(TmapCache*);

pds_status tc_gemm_plain(TcContext& c, const uint16_t* A, const uint16_t* W, float* C, int M,
                         int N, int K, cudaStream_t st, std::string* err);
pds_status tc_gemm_qkv(TcContext& c, const uint16_t* A, const WeightRows& W, int M, int K,
                       const QkvEpilogue& e, cudaStream_t st, std::string* err);
pds_status tc_gemm_resid(TcContext& c, const uint16_t* A, const uint16_t* W, int M, int N, int K,
                         const ResidEpilogue& e, cudaStream_t st, std::string* err);
pds_status tc_gemm_swiglu(TcContext& c, const uint16_t* A, const WeightRows& W, int M, int K,
                          const SwigluEpilogue& e, cudaStream_t st, std::string* err);
// The plain GEMM with its scratch in a static device array instead of a
// caller buffer (allocates nothing); at most tc_gemm_noalloc_max_tiles()
// output tiles of 128 x 128.
size_t tc_gemm_noalloc_max_tiles();
// Read and clear the status word of the current device's static scratch
// (0 if the no-allocation GEMM has not run on this device).
pds_status tc_noalloc_take_status(uint32_t* flags, std::string* err);
pds_status tc_gemm_plain_noalloc(const uint16_t* A, const uint16_t* W, float* C, int M, int N,
                                 int K, int num_sms, cudaStream_t st, std::string* err);
// Tensor map of a row-major bf16 matrix [outer, inner]: boxes of 64 columns
// (128 bytes, 128-byte swizzle) x box_rows rows; cached in c.maps.
// Launch facts of a kernel on the current device, made once per (kernel,
// device) with that device current (function attributes and occupancy are
// per device): the dynamic shared-memory limit of `fn`, and how many
// clusters of `cs` CTAs of `fn` launched with `cfg` fit on the GPU at once
// (0 if the query fails).
cudaError_t kernel_smem_attr(const void* fn, int bytes);
int kernel_max_clusters(const void* fn, const cudaLaunchConfig_t& cfg, int cs);
pds_status tc_map_bf16(TcContext& c, CUtensorMap* out, const void* p, uint64_t inner,
                       uint64_t outer, uint32_t box_rows, std::string* err);
// GQA causal attention on the tcgen05 tensor cores (head_dim 64 or 128).
// Attention scratch: bytes per unit of the chunked mode, and the most a call
// with batch B over an s-row prefix can use (chunked key ranges are used
// only as far as the scratch given in TcContext holds them).
size_t tc_attention_unit_bytes(int hd);
size_t tc_attention_scratch_bytes(int B, int s, int H, int hd);
// softcap > 0 caps the scaled scores (softcap * tanh(z / softcap)); window
// > 0 lets the row at position p see keys p - window < j <= p only.
pds_status tc_attention(TcContext& c, const uint16_t* q, const uint16_t* k, const uint16_t* v,
                        uint16_t* o, int B, int start_pos, int H, int Hkv, int hd, float softcap,
                        int window, cudaStream_t st, std::string* err);

}  // namespace pds
