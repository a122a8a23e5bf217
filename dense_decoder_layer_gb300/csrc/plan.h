// Plan and workspace layout of the dense prefill stack (host side).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <string>
#include <vector>

#include "../../include/pds.h"

namespace pds {

struct TmapCache;

struct Plan {
  pds_dims dims{};  // freq_factors is not kept (see omega)
  int q_width = 0, kv_width = 0;
  // Run-wide RoPE and attention options, resolved from dims.
  int rope_layout = PDS_ROPE_NEOX;
  int rot_dim = 0;               // rotated channels per head (<= head_dim)
  std::vector<double> omega;     // [rot_dim / 2] angular frequencies, float64
  float rope_mscale = 1.0f;
  float attn_softcap = 0.0f;     // 0: none
  int window = 0;                // 0: none
  // Device state made by pds_plan_create on the device current then (none
  // when the plan was made without a CUDA device).
  int device = -1;
  int num_sms = 0;
  uint32_t* d_status = nullptr;  // status word written by bounded device waits
  uint32_t* h_status = nullptr;  // pinned host copy of it, read after a stream synchronize
  TmapCache* maps = nullptr;  // encoded TMA descriptors, reused across calls
  // Per-kernel timing (pds_plan_set_timing).
  bool timing = false;
  struct Mark {
    int kind;
    cudaEvent_t start, stop;
  };
  std::vector<Mark> marks;          // recorded, not yet read
  std::vector<cudaEvent_t> events;  // free events
  int64_t launches[PDS_KERNEL_KINDS] = {};
  double total_ms[PDS_KERNEL_KINDS] = {};
  // CUDA graphs of recent call shapes: the whole call (every kernel of every
  // layer) is captured once per key (all pointers, start_pos, batch) and
  // replayed; at most kMaxGraphs are kept (least recently used goes).
  // PDS_GRAPH=0 turns this off (every call is enqueued kernel by kernel).
  static constexpr size_t kMaxGraphs = 4;
  bool graphs = true;
  struct Graph {
    std::vector<uintptr_t> key;
    cudaGraphExec_t exec = nullptr;
    uint64_t last_use = 0;
  };
  std::vector<Graph> graph_cache;
  uint64_t graph_clock = 0;
  cudaStream_t capture_stream = nullptr;
};

// Byte offsets into the caller's workspace.  total is the least a call
// needs; the attention's chunked key ranges use what lies beyond attn.
struct Layout {
  size_t x, h, a, ss_attn, ss_ffn, q, o, act, rope, gemm_ws, attn, total;
};

Layout make_layout(const Plan& p, int B);
// Bytes a call with batch <= B and start_pos <= s_max uses at most.
size_t workspace_bytes(const Plan& p, int B, int s_max);

// Scratch of the tensor-core GEMMs (stream-K partial tiles and tile
// counters) for a call with batch B.
size_t gemm_workspace_bytes(const Plan& p, int B);

pds_status enqueue_stack(Plan& p, const pds_layer* layers, uint16_t* const* k_cache,
                         uint16_t* const* v_cache, int start_pos, int B, const float* x_in,
                         float* x_out, char* ws, size_t ws_bytes, cudaStream_t st,
                         std::string* err);

// enqueue_stack through the plan's graph cache (or directly when graphs are off).
pds_status run_stack(Plan& p, const pds_layer* layers, uint16_t* const* k_cache,
                     uint16_t* const* v_cache, int start_pos, int B, const float* x_in,
                     float* x_out, char* ws, size_t ws_bytes, cudaStream_t st,
                     std::string* err);

// Make the plan's device state on the current device (pds_plan_create).
pds_status plan_attach_device(Plan& p, std::string* err);
pds_status plan_sync(Plan& p, cudaStream_t st, std::string* err);
pds_status plan_kernel_times(Plan& p, cudaStream_t st, pds_kernel_times* out, bool reset,
                             std::string* err);
void plan_release_device(Plan& p);

pds_status run_gemm_plain(const uint16_t* A, const uint16_t* W, float* C, int M, int N, int K,
                          char* ws, size_t ws_bytes, cudaStream_t st, std::string* err);
pds_status run_stuck_wait(uint32_t limit_us, cudaStream_t st, std::string* err);
// Synchronize and take (read and clear) the status words of the component
// entry points on the current device.
pds_status component_sync(cudaStream_t st, std::string* err);
// Address of the component entry points' status word on the current device.
uint32_t* component_status(std::string* err);
pds_status run_attention(const uint16_t* q, const uint16_t* k, const uint16_t* v, uint16_t* o,
                         int B, int start_pos, int H, int Hkv, int hd, float softcap, int window,
                         char* ws, size_t ws_bytes, cudaStream_t st, std::string* err);

}  // namespace pds
