// The layer loop of one prefill call: which kernels run, on which
// buffers, in which order.
//
// Per call: the (cos, sin) table of the call's positions and the
// first-layer norm prep.  Per layer (the seven matmuls of
// frink-models 0.29.0 src/decoder/cuda_prefill.rs, module doc, with
// everything between them fused into their epilogues):
//   1. QKV GEMM   a . [wq;wk;wv]^T, row scale of the attention RMSNorm,
//                 RoPE, q -> workspace, k/v -> cache rows [s, s+B)
//   2. attention  GQA causal over cache rows [0, s+B)
//   3. wo GEMM    h = x + o . wo^T, a = bf16(h * g_ffn), sum-of-squares
//   4. gate/up    act = silu(r * a.wg^T) * (r * a.wu^T)
//   5. down GEMM  x' = h + act . wd^T, a = bf16(x' * g_attn[l+1]), sum-of-squares
// The residual stream stays float32 throughout.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <string>

#include "common.cuh"
#include "kernels.h"
#include "plan.h"
#include "tc.h"

namespace pds {
namespace {

pds_status check_launch(const char* what, std::string* err) {
  cudaError_t ce = cudaGetLastError();
  if (ce != cudaSuccess) {
    *err = std::string(what) + ": " + cudaGetErrorString(ce);
    return PDS_ELAUNCH;
  }
  return PDS_OK;
}

// The plan's device state, made on the current device by pds_plan_create;
// every call must run with that device current.
pds_status check_device_state(const Plan& p, std::string* err) {
  if (!p.d_status) {
    *err = "the plan has no device state (it was created without a CUDA device)";
    return PDS_ELAUNCH;
  }
  int dev = -1;
  cudaError_t ce = cudaGetDevice(&dev);
  if (ce != cudaSuccess) {
    *err = std::string("no CUDA device: ") + cudaGetErrorString(ce);
    return PDS_ELAUNCH;
  }
  if (dev != p.device) {
    *err = "plan used on device " + std::to_string(dev) + ", created on device " +
           std::to_string(p.device);
    return PDS_EINVAL;
  }
  return PDS_OK;
}

// Status word of the component entry points (no plan).
__device__ uint32_t g_component_status;

int current_num_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

}  // namespace

uint32_t* component_status(std::string* err) {
  void* p = nullptr;
  cudaError_t ce = cudaGetSymbolAddress(&p, g_component_status);
  if (ce != cudaSuccess) {
    *err = std::string("status word address: ") + cudaGetErrorString(ce);
    return nullptr;
  }
  return static_cast<uint32_t*>(p);
}

pds_status component_sync(cudaStream_t st, std::string* err) {
  cudaError_t ce = cudaStreamSynchronize(st);
  if (ce != cudaSuccess) {
    *err = std::string("stream synchronize: ") + cudaGetErrorString(ce);
    return PDS_ELAUNCH;
  }
  uint32_t flags = 0;
  ce = cudaMemcpyFromSymbol(&flags, g_component_status, sizeof(flags));
  if (ce == cudaSuccess && flags) {
    const uint32_t zero = 0;
    ce = cudaMemcpyToSymbol(g_component_status, &zero, sizeof(zero));
  }
  if (ce != cudaSuccess) {
    *err = std::string("component status word: ") + cudaGetErrorString(ce);
    return PDS_ELAUNCH;
  }
  uint32_t noalloc_flags = 0;
  pds_status rc = tc_noalloc_take_status(&noalloc_flags, err);
  if (rc != PDS_OK) return rc;
  flags |= noalloc_flags;
  if (flags & kStatusTimeout) {
    *err = "a bounded device wait of a component call gave up (status word " +
           std::to_string(flags) + ")";
    return PDS_ETIMEOUT;
  }
  if (flags) {
    *err = "component status word " + std::to_string(flags);
    return PDS_ELAUNCH;
  }
  return PDS_OK;
}

pds_status plan_attach_device(Plan& p, std::string* err) {
  int dev = -1;
  cudaError_t ce = cudaGetDevice(&dev);
  if (ce == cudaSuccess)
    ce = cudaDeviceGetAttribute(&p.num_sms, cudaDevAttrMultiProcessorCount, dev);
  if (ce == cudaSuccess) ce = cudaMalloc(&p.d_status, sizeof(uint32_t));
  if (ce == cudaSuccess) ce = cudaMemset(p.d_status, 0, sizeof(uint32_t));
  if (ce == cudaSuccess) ce = cudaMallocHost(&p.h_status, sizeof(uint32_t));
  if (ce == cudaSuccess) ce = cudaStreamCreateWithFlags(&p.capture_stream, cudaStreamNonBlocking);
  if (ce != cudaSuccess) {
    *err = std::string("plan device state: ") + cudaGetErrorString(ce);
    plan_release_device(p);
    return PDS_ENOMEM;
  }
  *p.h_status = 0;
  p.device = dev;
  p.maps = tmap_cache_create();
  return PDS_OK;
}

size_t gemm_workspace_bytes(const Plan& p, int B) {
  const int n_qkv = p.q_width + 2 * p.kv_width;
  const int max_n = std::max(std::max(n_qkv, 2 * p.dims.ffn_dim), p.dims.d_model);
  return tc_gemm_scratch_bytes(B, (max_n + 127) / 128);
}

void plan_release_device(Plan& p) {
  for (Plan::Graph& g : p.graph_cache)
    if (g.exec) cudaGraphExecDestroy(g.exec);
  p.graph_cache.clear();
  if (p.capture_stream) cudaStreamDestroy(p.capture_stream);
  p.capture_stream = nullptr;
  for (const Plan::Mark& m : p.marks) {
    cudaEventDestroy(m.start);
    cudaEventDestroy(m.stop);
  }
  for (cudaEvent_t e : p.events) cudaEventDestroy(e);
  p.marks.clear();
  p.events.clear();
  if (p.d_status) cudaFree(p.d_status);
  p.d_status = nullptr;
  if (p.h_status) cudaFreeHost(p.h_status);
  p.h_status = nullptr;
  if (p.maps) tmap_cache_destroy(p.maps);
  p.maps = nullptr;
}

pds_status plan_sync(Plan& p, cudaStream_t st, std::string* err) {
  // the status word comes back on the stream, behind the call's work, so
  // that one synchronize covers both
  cudaError_t ce = cudaSuccess;
  if (p.d_status && p.h_status)
    ce = cudaMemcpyAsync(p.h_status, p.d_status, sizeof(uint32_t), cudaMemcpyDeviceToHost, st);
  if (ce == cudaSuccess) ce = cudaStreamSynchronize(st);
  if (ce != cudaSuccess) {
    *err = std::string("stream synchronize: ") + cudaGetErrorString(ce);
    return PDS_ELAUNCH;
  }
  if (!p.d_status || !p.h_status) return PDS_OK;
  const uint32_t flags = *static_cast<volatile uint32_t*>(p.h_status);
  if (flags) {
    *p.h_status = 0;
    ce = cudaMemset(p.d_status, 0, sizeof(uint32_t));
  }
  if (ce != cudaSuccess) {
    *err = std::string("status word: ") + cudaGetErrorString(ce);
    return PDS_ELAUNCH;
  }
  if (flags & kStatusTimeout) {
    *err = "a bounded device wait gave up (status word " + std::to_string(flags) + ")";
    return PDS_ETIMEOUT;
  }
  if (flags) {
    *err = "device status word " + std::to_string(flags);
    return PDS_ELAUNCH;
  }
  return PDS_OK;
}

pds_status enqueue_stack(Plan& p, const pds_layer* layers, uint16_t* const* k_cache,
                         uint16_t* const* v_cache, int s, int B, const float* x_in, float* x_out,
                         char* ws, size_t ws_bytes, cudaStream_t st, std::string* err) {
  pds_status rc = check_device_state(p, err);
  if (rc != PDS_OK) return rc;
  const pds_dims& D = p.dims;
  const int d = D.d_model, F = D.ffn_dim, hd = D.head_dim, L = D.n_layers;
  const Layout lay = make_layout(p, B);
  float* X = reinterpret_cast<float*>(ws + lay.x);
  float* Hs = reinterpret_cast<float*>(ws + lay.h);
  uint16_t* A = reinterpret_cast<uint16_t*>(ws + lay.a);
  float* ss_attn = reinterpret_cast<float*>(ws + lay.ss_attn);
  float* ss_ffn = reinterpret_cast<float*>(ws + lay.ss_ffn);
  uint16_t* Q = reinterpret_cast<uint16_t*>(ws + lay.q);
  uint16_t* O = reinterpret_cast<uint16_t*>(ws + lay.o);
  uint16_t* ACT = reinterpret_cast<uint16_t*>(ws + lay.act);
  float2* rope = reinterpret_cast<float2*>(ws + lay.rope);
  const int parts = d / 64;
  const float inv_d = 1.0f / (float)d;

  // Per-kernel timing marks (pds_plan_set_timing): events on the call's stream.
  auto mark = [&](int kind) -> Plan::Mark* {
    if (!p.timing) return nullptr;
    Plan::Mark m{kind, nullptr, nullptr};
    for (cudaEvent_t* e : {&m.start, &m.stop}) {
      if (!p.events.empty()) {
        *e = p.events.back();
        p.events.pop_back();
      } else if (cudaEventCreate(e) != cudaSuccess) {
        return nullptr;
      }
    }
    p.marks.push_back(m);
    cudaEventRecord(m.start, st);
    return &p.marks.back();
  };
  auto done = [&](Plan::Mark* m) {
    if (m) cudaEventRecord(m->stop, st);
  };

  // the plan's float64 angular frequencies of the rotated pairs
  RopeFreqs rf{};
  rf.n_pairs = p.rot_dim / 2;
  rf.mscale = p.rope_mscale;
  for (int i = 0; i < rf.n_pairs; ++i) rf.omega[i] = p.omega[i];

  Plan::Mark* mk = mark(PDS_KERNEL_PREP);
  launch_rope_table(rope, B, s, rf, st);
  launch_norm_prep(x_in, layers[0].attn_norm_w, A, ss_attn, B, d, st);
  done(mk);
  if ((rc = check_launch("norm prep", err)) != PDS_OK) return rc;

  TcContext tc{};
  tc.num_sms = p.num_sms;
  tc.status = p.d_status;
  tc.ws = ws + lay.gemm_ws;
  tc.ws_bytes = gemm_workspace_bytes(p, B);
  tc.maps = p.maps;
  tc.pdl = true;
  tc.attn_ws = ws + lay.attn;
  tc.attn_ws_bytes = ws_bytes > lay.attn ? ws_bytes - lay.attn : 0;
  {
    // stream-K tile counters start at zero; every GEMM leaves them at zero
    const size_t part = tc_gemm_scratch_bytes(B, 0);
    cudaError_t ce = cudaMemsetAsync(tc.ws + part, 0, tc.ws_bytes - part, st);
    if (ce != cudaSuccess) {
      *err = std::string("tile counter reset: ") + cudaGetErrorString(ce);
      return PDS_ELAUNCH;
    }
  }

  for (int l = 0; l < L; ++l) {
    const pds_layer& w = layers[l];
    const float* x_cur = (l == 0) ? x_in : X;
    float* x_next = (l == L - 1) ? x_out : X;
    const float* g_next = (l == L - 1) ? nullptr : layers[l + 1].attn_norm_w;

    QkvEpilogue qe{};
    qe.rs = RowScale{ss_attn, parts, inv_d, D.rms_eps};
    qe.rope = rope;
    qe.rope_ld = B;
    qe.q = Q;
    qe.k_cache = k_cache[l];
    qe.v_cache = v_cache[l];
    qe.start_pos = s;
    qe.q_width = p.q_width;
    qe.kv_width = p.kv_width;
    qe.head_dim = hd;
    qe.rope_layout = p.rope_layout;
    qe.rot_dim = p.rot_dim;
    qe.bias[0] = w.q_bias;
    qe.bias[1] = w.k_bias;
    qe.bias[2] = w.v_bias;
    qe.norm[0] = w.q_norm;
    qe.norm[1] = w.k_norm;
    WeightRows wqkv{{w.wq, w.wk, w.wv}, {p.q_width, p.kv_width, p.kv_width}, 3};

    ResidEpilogue oe{x_cur, Hs, w.ffn_norm_w, A, ss_ffn};
    SwigluEpilogue ge{RowScale{ss_ffn, parts, inv_d, D.rms_eps}, ACT, F};
    WeightRows wgu{{w.w_gate, w.w_up, nullptr}, {F, F, 0}, 2};
    ResidEpilogue de{Hs, x_next, g_next, A, ss_attn};

    mk = mark(PDS_KERNEL_QKV);
    rc = tc_gemm_qkv(tc, A, wqkv, B, d, qe, st, err);
    done(mk);
    if (rc != PDS_OK) return rc;
    mk = mark(PDS_KERNEL_ATTN);
    rc = tc_attention(tc, Q, k_cache[l], v_cache[l], O, B, s, D.n_heads, D.n_kv_heads, hd,
                      p.attn_softcap, p.window, st, err);
    done(mk);
    if (rc != PDS_OK) return rc;
    mk = mark(PDS_KERNEL_WO);
    rc = tc_gemm_resid(tc, O, w.wo, B, d, p.q_width, oe, st, err);
    done(mk);
    if (rc != PDS_OK) return rc;
    mk = mark(PDS_KERNEL_GATEUP);
    rc = tc_gemm_swiglu(tc, A, wgu, B, d, ge, st, err);
    done(mk);
    if (rc != PDS_OK) return rc;
    mk = mark(PDS_KERNEL_DOWN);
    rc = tc_gemm_resid(tc, ACT, w.w_down, B, d, F, de, st, err);
    done(mk);
    if (rc != PDS_OK) return rc;
  }
  return PDS_OK;
}

pds_status run_stack(Plan& p, const pds_layer* layers, uint16_t* const* k_cache,
                     uint16_t* const* v_cache, int s, int B, const float* x_in, float* x_out,
                     char* ws, size_t ws_bytes, cudaStream_t st, std::string* err) {
  if (!p.graphs || p.timing)
    return enqueue_stack(p, layers, k_cache, v_cache, s, B, x_in, x_out, ws, ws_bytes, st, err);
  pds_status rc = check_device_state(p, err);
  if (rc != PDS_OK) return rc;
  std::vector<uintptr_t> key;
  key.reserve(8 + 16 * p.dims.n_layers);
  key.push_back(static_cast<uintptr_t>(s));
  key.push_back(static_cast<uintptr_t>(B));
  key.push_back(reinterpret_cast<uintptr_t>(x_in));
  key.push_back(reinterpret_cast<uintptr_t>(x_out));
  key.push_back(reinterpret_cast<uintptr_t>(ws));
  key.push_back(static_cast<uintptr_t>(ws_bytes));
  for (int l = 0; l < p.dims.n_layers; ++l) {
    const pds_layer& w = layers[l];
    for (const void* q : {(const void*)w.attn_norm_w, (const void*)w.ffn_norm_w,
                          (const void*)w.wq, (const void*)w.wk, (const void*)w.wv,
                          (const void*)w.wo, (const void*)w.w_gate, (const void*)w.w_up,
                          (const void*)w.w_down, (const void*)k_cache[l], (const void*)v_cache[l],
                          (const void*)w.q_bias, (const void*)w.k_bias, (const void*)w.v_bias,
                          (const void*)w.q_norm, (const void*)w.k_norm})
      key.push_back(reinterpret_cast<uintptr_t>(q));
  }
  Plan::Graph* hit = nullptr;
  for (Plan::Graph& g : p.graph_cache)
    if (g.key == key) hit = &g;
  if (!hit) {
    cudaError_t ce = cudaStreamBeginCapture(p.capture_stream, cudaStreamCaptureModeRelaxed);
    if (ce != cudaSuccess) {
      *err = std::string("graph capture start: ") + cudaGetErrorString(ce);
      return PDS_ELAUNCH;
    }
    rc = enqueue_stack(p, layers, k_cache, v_cache, s, B, x_in, x_out, ws, ws_bytes,
                       p.capture_stream, err);
    cudaGraph_t graph = nullptr;
    ce = cudaStreamEndCapture(p.capture_stream, &graph);
    if (rc != PDS_OK || ce != cudaSuccess) {
      if (graph) cudaGraphDestroy(graph);
      if (rc == PDS_OK) {
        *err = std::string("graph capture: ") + cudaGetErrorString(ce);
        rc = PDS_ELAUNCH;
      }
      cudaGetLastError();
      return rc;
    }
    cudaGraphExec_t exec = nullptr;
    ce = cudaGraphInstantiate(&exec, graph, 0);
    cudaGraphDestroy(graph);
    if (ce != cudaSuccess) {
      *err = std::string("graph instantiate: ") + cudaGetErrorString(ce);
      return PDS_ELAUNCH;
    }
    if (p.graph_cache.size() >= Plan::kMaxGraphs) {
      auto lru = std::min_element(p.graph_cache.begin(), p.graph_cache.end(),
                                  [](const Plan::Graph& a, const Plan::Graph& b) {
                                    return a.last_use < b.last_use;
                                  });
      cudaGraphExecDestroy(lru->exec);
      p.graph_cache.erase(lru);
    }
    p.graph_cache.push_back(Plan::Graph{std::move(key), exec, 0});
    hit = &p.graph_cache.back();
  }
  hit->last_use = ++p.graph_clock;
  cudaError_t ce = cudaGraphLaunch(hit->exec, st);
  if (ce != cudaSuccess) {
    *err = std::string("graph launch: ") + cudaGetErrorString(ce);
    return PDS_ELAUNCH;
  }
  return PDS_OK;
}

pds_status plan_kernel_times(Plan& p, cudaStream_t st, pds_kernel_times* out, bool reset,
                             std::string* err) {
  cudaError_t ce = cudaStreamSynchronize(st);
  if (ce != cudaSuccess) {
    *err = std::string("stream synchronize: ") + cudaGetErrorString(ce);
    return PDS_ELAUNCH;
  }
  for (const Plan::Mark& m : p.marks) {
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, m.start, m.stop) == cudaSuccess) {
      p.launches[m.kind] += 1;
      p.total_ms[m.kind] += ms;
    }
    p.events.push_back(m.start);
    p.events.push_back(m.stop);
  }
  p.marks.clear();
  for (int k = 0; k < PDS_KERNEL_KINDS; ++k) {
    out->launches[k] = p.launches[k];
    out->total_ms[k] = p.total_ms[k];
    if (reset) {
      p.launches[k] = 0;
      p.total_ms[k] = 0.0;
    }
  }
  return PDS_OK;
}

pds_status run_attention(const uint16_t* q, const uint16_t* k, const uint16_t* v, uint16_t* o,
                         int B, int start_pos, int H, int Hkv, int hd, float softcap, int window,
                         char* ws, size_t ws_bytes, cudaStream_t st, std::string* err) {
  TcContext tc{};
  tc.num_sms = current_num_sms();
  tc.attn_ws = ws;
  tc.attn_ws_bytes = ws_bytes;
  if (!(tc.status = component_status(err))) return PDS_ELAUNCH;
  pds_status rc =
      tc_attention(tc, q, k, v, o, B, start_pos, H, Hkv, hd, softcap, window, st, err);
  if (rc == PDS_OK) rc = check_launch("attention", err);
  return rc;
}

pds_status run_gemm_plain(const uint16_t* A, const uint16_t* W, float* C, int M, int N, int K,
                          char* ws, size_t ws_bytes, cudaStream_t st, std::string* err) {
  TcContext tc{};
  tc.num_sms = current_num_sms();
  if (!(tc.status = component_status(err))) return PDS_ELAUNCH;
  tc.ws = ws;
  tc.ws_bytes = ws_bytes;
  const size_t part = tc_gemm_scratch_bytes(M, 0);
  cudaError_t ce = cudaMemsetAsync(ws + part, 0, ws_bytes - part, st);
  if (ce != cudaSuccess) {
    *err = std::string("tile counter reset: ") + cudaGetErrorString(ce);
    return PDS_ELAUNCH;
  }
  return tc_gemm_plain(tc, A, W, C, M, N, K, st, err);
}

}  // namespace pds
