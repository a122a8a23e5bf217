// Host side of the C ABI: validation and declines, workspace layout, the
// per-call enqueue of the layer loop, error reporting.
//
// The call shape follows frink-models 0.29.0 src/decoder/cuda_prefill.rs
// (try_cuda_prefill_dense_stack / cuda_prefill_layer): refusals are
// decided on the host before any device work; one enqueue covers the whole
// run of layers; the hidden batch crosses host<->device once each way; a
// failure after admission is reported once per distinct message.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <set>
#include <string>
#include <vector>

#include "../../include/pds.h"
#include "kernels.h"
#include "plan.h"
#include "tc.h"

namespace {

thread_local std::string t_last_error;

void warn_once(const std::string& msg) {
  static std::mutex mu;
  static std::set<std::string> seen;
  std::lock_guard<std::mutex> g(mu);
  if (seen.insert(msg).second) std::fprintf(stderr, "%s\n", msg.c_str());
}

pds_status fail(pds_status st, const std::string& msg) {
  t_last_error = msg;
  if (st == PDS_ELAUNCH || st == PDS_ETIMEOUT || st == PDS_ENOMEM)
    warn_once("pds: prefill stack failed after admission: " + msg);
  return st;
}

bool env_flag(const char* name) {
  const char* v = std::getenv(name);
  return v && *v && std::strcmp(v, "0") != 0;
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

namespace pds {

Layout make_layout(const Plan& p, int B) {
  Layout L{};
  size_t off = 0;
  auto take = [&](size_t bytes) {
    size_t o = off;
    off = align_up(off + bytes, 256);
    return o;
  };
  const size_t Bz = (size_t)B;
  const int d = p.dims.d_model;
  L.x = take(Bz * d * 4);
  L.h = take(Bz * d * 4);
  L.a = take(Bz * d * 2);
  L.ss_attn = take(Bz * (d / 64) * 4);
  L.ss_ffn = take(Bz * (d / 64) * 4);
  L.q = take(Bz * p.q_width * 2);
  L.o = take(Bz * p.q_width * 2);
  L.act = take(Bz * p.dims.ffn_dim * 2);
  L.rope = take(Bz * (p.dims.head_dim / 2) * 8);
  L.gemm_ws = take(gemm_workspace_bytes(p, B));
  L.attn = off;
  L.total = off;
  return L;
}

size_t workspace_bytes(const Plan& p, int B, int s_max) {
  const Layout L = make_layout(p, B);
  return L.attn + align_up(tc_attention_scratch_bytes(B, s_max, p.dims.n_heads,
                                                      p.dims.head_dim), 256);
}

}  // namespace pds

using pds::Plan;

struct pds_plan : Plan {};

extern "C" {

const char* pds_last_error(void) { return t_last_error.c_str(); }

pds_status pds_plan_create(const pds_dims* dims, pds_plan** out) {
  if (!out) return fail(PDS_EINVAL, "pds_plan_create: out is NULL");
  *out = nullptr;
  if (!dims) return fail(PDS_EINVAL, "pds_plan_create: dims is NULL");
  const pds_dims& d = *dims;
  if (d.n_layers < 1 || d.d_model < 1 || d.n_heads < 1 || d.n_kv_heads < 1 || d.head_dim < 1 ||
      d.ffn_dim < 1)
    return fail(PDS_EINVAL, "pds_plan_create: every dimension must be positive");
  if (!(d.rope_theta > 0.f) || !(d.rms_eps >= 0.f) || !std::isfinite(d.rope_theta) ||
      !std::isfinite(d.rms_eps))
    return fail(PDS_EINVAL, "pds_plan_create: rope_theta must be > 0 and rms_eps >= 0");
  if (env_flag("PDS_DISABLE")) return fail(PDS_DECLINED, "declined: PDS_DISABLE is set");
  if (d.n_heads % d.n_kv_heads != 0)
    return fail(PDS_DECLINED, "declined: n_heads is not a multiple of n_kv_heads");
  if (d.head_dim != 64 && d.head_dim != 128)
    return fail(PDS_DECLINED, "declined: head_dim must be 64 or 128");
  if (d.d_model % 128 != 0 || d.ffn_dim % 128 != 0)
    return fail(PDS_DECLINED, "declined: d_model and ffn_dim must be multiples of 128");
  if ((d.n_heads * d.head_dim) % 128 != 0 || (d.n_kv_heads * d.head_dim) % 128 != 0)
    return fail(PDS_DECLINED, "declined: n_heads*head_dim and n_kv_heads*head_dim must be multiples of 128");
  // run-wide RoPE and attention options
  if (d.rope_layout != PDS_ROPE_NEOX && d.rope_layout != PDS_ROPE_NORM)
    return fail(PDS_EINVAL, "pds_plan_create: rope_layout must be PDS_ROPE_NEOX or PDS_ROPE_NORM");
  if (d.rot_dim < 0 || d.rot_dim > d.head_dim || d.rot_dim % 2)
    return fail(PDS_EINVAL, "pds_plan_create: rot_dim must be 0 or even and <= head_dim");
  const int rot = d.rot_dim ? d.rot_dim : d.head_dim;
  if (rot % (d.rope_layout == PDS_ROPE_NEOX ? 32 : 16) != 0)
    return fail(PDS_DECLINED, "declined: rot_dim must be a multiple of 32 (Neox) or 16 (Norm)");
  if (!std::isfinite(d.rope_mscale) || d.rope_mscale < 0.f)
    return fail(PDS_EINVAL, "pds_plan_create: rope_mscale must be 0 or > 0");
  if (!std::isfinite(d.attn_softcap) || d.attn_softcap < 0.f)
    return fail(PDS_EINVAL, "pds_plan_create: attn_softcap must be 0 or > 0");
  if (d.window < 0) return fail(PDS_EINVAL, "pds_plan_create: window must be >= 0");
  if (d.freq_factors)
    for (int i = 0; i < rot / 2; ++i)
      if (!(d.freq_factors[i] > 0.f) || !std::isfinite(d.freq_factors[i]))
        return fail(PDS_EINVAL, "pds_plan_create: freq_factors must be finite and > 0");
  pds_plan* p = new (std::nothrow) pds_plan();
  if (!p) return fail(PDS_ENOMEM, "pds_plan_create: out of host memory");
  p->dims = d;
  p->dims.freq_factors = nullptr;  // the caller's array is not kept
  p->q_width = d.n_heads * d.head_dim;
  p->kv_width = d.n_kv_heads * d.head_dim;
  p->rope_layout = d.rope_layout;
  p->rot_dim = rot;
  // omega_i = theta^(-2i/rot_dim) / freq_factors[i], in float64
  // (cuda_prefill.rs, LayerRopeCuda: theta, freq_factors, rot_dim)
  p->omega.resize(rot / 2);
  for (int i = 0; i < rot / 2; ++i)
    p->omega[i] = std::pow(static_cast<double>(d.rope_theta), -2.0 * i / rot) /
                  (d.freq_factors ? static_cast<double>(d.freq_factors[i]) : 1.0);
  p->rope_mscale = d.rope_mscale > 0.f ? d.rope_mscale : 1.0f;
  p->attn_softcap = d.attn_softcap;
  p->window = d.window;
  const char* g = std::getenv("PDS_GRAPH");
  p->graphs = !(g && std::strcmp(g, "0") == 0);
  // The plan's device state, on the current device, once the shape is
  // admitted; without a CUDA device the plan stays host-only.
  int ndev = 0;
  if (cudaGetDeviceCount(&ndev) == cudaSuccess && ndev > 0) {
    std::string err;
    const pds_status st = pds::plan_attach_device(*p, &err);
    if (st != PDS_OK) {
      delete p;
      return fail(st, err);
    }
  } else {
    cudaGetLastError();
  }
  *out = p;
  return PDS_OK;
}

void pds_plan_destroy(pds_plan* plan) {
  if (!plan) return;
  pds::plan_release_device(*plan);
  delete plan;
}

size_t pds_workspace_bytes(const pds_plan* plan, int32_t max_batch, int32_t max_start_pos) {
  if (!plan || max_batch < 1 || max_start_pos < 0) return 0;
  return pds::workspace_bytes(*plan, max_batch, max_start_pos);
}

static pds_status check_call(pds_plan* plan, const pds_layer* layers, uint16_t* const* kc,
                             uint16_t* const* vc, int32_t cap, int32_t s, int32_t B,
                             const void* in, const void* out, void* ws, size_t ws_bytes,
                             bool device_io) {
  if (!plan) return fail(PDS_EINVAL, "plan is NULL");
  if (!layers || !kc || !vc) return fail(PDS_EINVAL, "layers / k_cache / v_cache is NULL");
  if (!in || !out) return fail(PDS_EINVAL, "hidden_in / hidden_out is NULL");
  if (B < 1) return fail(PDS_EINVAL, "batch must be >= 1");
  if (s < 0) return fail(PDS_EINVAL, "start_pos must be >= 0");
  if ((int64_t)s + B > cap)
    return fail(PDS_DECLINED, "declined: start_pos + batch exceeds the cache capacity");
  if (!ws) return fail(PDS_EINVAL, "workspace is NULL");
  if (!aligned16(ws)) return fail(PDS_EINVAL, "workspace is not 16-byte aligned");
  if (ws_bytes < pds::make_layout(*plan, B).total)
    return fail(PDS_EINVAL, "workspace is smaller than pds_workspace_bytes(plan, batch, 0)");
  if (device_io && (!aligned16(in) || !aligned16(out)))
    return fail(PDS_EINVAL, "device hidden_in / hidden_out not 16-byte aligned");
  for (int l = 0; l < plan->dims.n_layers; ++l) {
    const pds_layer& w = layers[l];
    const void* ptrs[] = {w.attn_norm_w, w.ffn_norm_w, w.wq, w.wk, w.wv,
                          w.wo,          w.w_gate,     w.w_up, w.w_down, kc[l], vc[l]};
    for (const void* q : ptrs) {
      if (!q) return fail(PDS_EINVAL, "layer " + std::to_string(l) + ": NULL weight or cache");
      if (!aligned16(q))
        return fail(PDS_EINVAL, "layer " + std::to_string(l) + ": pointer not 16-byte aligned");
    }
    for (const void* q : {(const void*)w.q_bias, (const void*)w.k_bias, (const void*)w.v_bias,
                          (const void*)w.q_norm, (const void*)w.k_norm})
      if (q && !aligned16(q))
        return fail(PDS_EINVAL,
                    "layer " + std::to_string(l) + ": extra (bias / norm) not 16-byte aligned");
  }
  // Fault injection for the callers' failure handling: the call is admitted,
  // then fails as a launch would, before any device work.
  if (env_flag("PDS_FAULT_AFTER_ADMIT"))
    return fail(PDS_ELAUNCH, "injected failure after admission (PDS_FAULT_AFTER_ADMIT)");
  return PDS_OK;
}

pds_status pds_prefill_dense_stack_device(pds_plan* plan, const pds_layer* layers,
                                          uint16_t* const* k_cache, uint16_t* const* v_cache,
                                          int32_t cache_capacity, int32_t start_pos,
                                          int32_t batch, const float* hidden_in_dev,
                                          float* hidden_out_dev, void* workspace,
                                          size_t workspace_bytes, void* stream) {
  pds_status st = check_call(plan, layers, k_cache, v_cache, cache_capacity, start_pos, batch,
                             hidden_in_dev, hidden_out_dev, workspace, workspace_bytes, true);
  if (st != PDS_OK) return st;
  std::string err;
  st = pds::run_stack(*plan, layers, k_cache, v_cache, start_pos, batch, hidden_in_dev,
                      hidden_out_dev, static_cast<char*>(workspace), workspace_bytes,
                      static_cast<cudaStream_t>(stream), &err);
  if (st != PDS_OK) return fail(st, err);
  return PDS_OK;
}

pds_status pds_prefill_dense_stack(pds_plan* plan, const pds_layer* layers,
                                   uint16_t* const* k_cache, uint16_t* const* v_cache,
                                   int32_t cache_capacity, int32_t start_pos, int32_t batch,
                                   const float* hidden_in, float* hidden_out, void* workspace,
                                   size_t workspace_bytes, void* stream) {
  pds_status st = check_call(plan, layers, k_cache, v_cache, cache_capacity, start_pos, batch,
                             hidden_in, hidden_out, workspace, workspace_bytes, false);
  if (st != PDS_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const pds::Layout lay = pds::make_layout(*plan, batch);
  float* xdev = reinterpret_cast<float*>(static_cast<char*>(workspace) + lay.x);
  const size_t bytes = (size_t)batch * plan->dims.d_model * sizeof(float);
  cudaError_t ce = cudaMemcpyAsync(xdev, hidden_in, bytes, cudaMemcpyHostToDevice, s);
  if (ce != cudaSuccess)
    return fail(PDS_ELAUNCH, std::string("upload of hidden_in: ") + cudaGetErrorString(ce));
  std::string err;
  st = pds::run_stack(*plan, layers, k_cache, v_cache, start_pos, batch, xdev, xdev,
                      static_cast<char*>(workspace), workspace_bytes, s, &err);
  if (st != PDS_OK) return fail(st, err);
  ce = cudaMemcpyAsync(hidden_out, xdev, bytes, cudaMemcpyDeviceToHost, s);
  if (ce != cudaSuccess)
    return fail(PDS_ELAUNCH, std::string("download of hidden_out: ") + cudaGetErrorString(ce));
  return pds_plan_sync(plan, stream);
}

pds_status pds_plan_sync(pds_plan* plan, void* stream) {
  if (!plan) return fail(PDS_EINVAL, "plan is NULL");
  std::string err;
  pds_status st = pds::plan_sync(*plan, static_cast<cudaStream_t>(stream), &err);
  if (st != PDS_OK) return fail(st, err);
  return PDS_OK;
}

pds_status pds_selftest_stuck_wait(uint32_t limit_us, void* stream) {
  if (limit_us == 0 || limit_us > 10000000u)
    return fail(PDS_EINVAL, "pds_selftest_stuck_wait: limit_us must be in (0, 10 s]");
  std::string err;
  pds_status st = pds::run_stuck_wait(limit_us, static_cast<cudaStream_t>(stream), &err);
  if (st != PDS_OK) return fail(st, err);
  return PDS_OK;
}

pds_status pds_component_sync(void* stream) {
  std::string err;
  pds_status st = pds::component_sync(static_cast<cudaStream_t>(stream), &err);
  if (st == PDS_ETIMEOUT) {
    t_last_error = err;  // reported to the caller, who asked for it
    return st;
  }
  if (st != PDS_OK) return fail(st, err);
  return PDS_OK;
}

pds_status pds_plan_set_timing(pds_plan* plan, int32_t enable) {
  if (!plan) return fail(PDS_EINVAL, "plan is NULL");
  plan->timing = enable != 0;
  return PDS_OK;
}

pds_status pds_plan_kernel_times(pds_plan* plan, void* stream, pds_kernel_times* out,
                                 int32_t reset) {
  if (!plan || !out) return fail(PDS_EINVAL, "plan or out is NULL");
  std::string err;
  pds_status st =
      pds::plan_kernel_times(*plan, static_cast<cudaStream_t>(stream), out, reset != 0, &err);
  if (st != PDS_OK) return fail(st, err);
  return PDS_OK;
}

size_t pds_gemm_workspace_bytes(int32_t M, int32_t N) {
  if (M < 1 || N < 1) return 0;
  return pds::tc_gemm_scratch_bytes(M, (N + 127) / 128);
}

pds_status pds_gemm_bf16(const uint16_t* A, const uint16_t* W, float* C, int32_t M, int32_t N,
                         int32_t K, void* workspace, size_t workspace_bytes, void* stream) {
  if (!A || !W || !C || !workspace) return fail(PDS_EINVAL, "pds_gemm_bf16: NULL operand");
  if (M < 1 || N < 128 || K < 64) return fail(PDS_EINVAL, "pds_gemm_bf16: bad size");
  if (N % 128 || K % 64)
    return fail(PDS_DECLINED, "declined: pds_gemm_bf16 needs N % 128 == 0 and K % 64 == 0");
  if (!aligned16(A) || !aligned16(W) || !aligned16(C) || !aligned16(workspace))
    return fail(PDS_EINVAL, "pds_gemm_bf16: operand not 16-byte aligned");
  if (workspace_bytes < pds_gemm_workspace_bytes(M, N))
    return fail(PDS_EINVAL, "pds_gemm_bf16: workspace smaller than pds_gemm_workspace_bytes");
  std::string err;
  pds_status st = pds::run_gemm_plain(A, W, C, M, N, K, static_cast<char*>(workspace),
                                      workspace_bytes, static_cast<cudaStream_t>(stream), &err);
  if (st != PDS_OK) return fail(st, err);
  return PDS_OK;
}

pds_status pds_gemm_bf16_noalloc(const uint16_t* A, const uint16_t* W, float* C, int32_t M,
                                 int32_t N, int32_t K, void* stream) {
  if (!A || !W || !C) return fail(PDS_EINVAL, "pds_gemm_bf16_noalloc: NULL operand");
  if (M < 1 || N < 128 || K < 64) return fail(PDS_EINVAL, "pds_gemm_bf16_noalloc: bad size");
  if (N % 128 || K % 64)
    return fail(PDS_DECLINED,
                "declined: pds_gemm_bf16_noalloc needs N % 128 == 0 and K % 64 == 0");
  if (!aligned16(A) || !aligned16(W) || !aligned16(C))
    return fail(PDS_EINVAL, "pds_gemm_bf16_noalloc: operand not 16-byte aligned");
  const size_t tiles = static_cast<size_t>((M + 127) / 128) * (N / 128);
  if (tiles > pds::tc_gemm_noalloc_max_tiles())
    return fail(PDS_EINVAL, "pds_gemm_bf16_noalloc: ceil(M/128) * (N/128) = " +
                                std::to_string(tiles) + " output tiles, more than the " +
                                std::to_string(pds::tc_gemm_noalloc_max_tiles()) +
                                " its static scratch holds");
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return fail(PDS_ELAUNCH, "pds_gemm_bf16_noalloc: no CUDA device");
  std::string err;
  pds_status st = pds::tc_gemm_plain_noalloc(A, W, C, M, N, K, sms,
                                             static_cast<cudaStream_t>(stream), &err);
  if (st != PDS_OK) return fail(st, err);
  return PDS_OK;
}

size_t pds_attention_workspace_bytes(int32_t batch, int32_t start_pos, int32_t n_heads,
                                     int32_t head_dim) {
  if (batch < 1 || start_pos < 0 || n_heads < 1 || (head_dim != 64 && head_dim != 128)) return 0;
  return pds::tc_attention_scratch_bytes(batch, start_pos, n_heads, head_dim);
}

pds_status pds_attention(const uint16_t* q, const uint16_t* k, const uint16_t* v, uint16_t* o,
                         int32_t batch, int32_t start_pos, int32_t n_heads, int32_t n_kv_heads,
                         int32_t head_dim, float softcap, int32_t window, void* workspace,
                         size_t workspace_bytes, void* stream) {
  if (!q || !k || !v || !o) return fail(PDS_EINVAL, "pds_attention: NULL operand");
  if (batch < 1 || start_pos < 0 || n_heads < 1 || n_kv_heads < 1)
    return fail(PDS_EINVAL, "pds_attention: bad size");
  if (!(softcap >= 0.f) || !std::isfinite(softcap) || window < 0)
    return fail(PDS_EINVAL, "pds_attention: softcap and window must be >= 0");
  if (n_heads % n_kv_heads != 0 || (head_dim != 64 && head_dim != 128))
    return fail(PDS_DECLINED, "declined: pds_attention needs H % Hkv == 0 and hd in {64, 128}");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) ||
      (workspace && !aligned16(workspace)))
    return fail(PDS_EINVAL, "pds_attention: operand not 16-byte aligned");
  if (!workspace) workspace_bytes = 0;
  std::string err;
  pds_status st = pds::run_attention(q, k, v, o, batch, start_pos, n_heads, n_kv_heads, head_dim,
                                     softcap, window, static_cast<char*>(workspace),
                                     workspace_bytes, static_cast<cudaStream_t>(stream), &err);
  if (st != PDS_OK) return fail(st, err);
  return PDS_OK;
}

}  // extern "C"
