/*
 * pds.h -- C ABI of the GB300 dense prefill stack.
 *
 * One call runs a batch of B new tokens through a run of L consecutive
 * dense Llama-style decoder layers on one GPU and returns the new hidden
 * batch plus every layer's new K/V rows.  Each layer computes
 *
 *     h  = x + wo(attn(rope(q,k), v))      q,k,v = rms_norm(x) . wq/wk/wv
 *     x' = h + down(silu(gate(m)) * up(m)), m     = rms_norm(h)
 *
 * (frink-models 0.49.0 src/fused_layer.rs, module doc "What it refuses":
 * the fused layer is exactly x + ffn(rms_norm(x + branch)) with a SwiGLU
 * FFN of one dense expert; frink-models 0.29.0
 * src/decoder/cuda_prefill.rs, module doc: the hidden batch goes up once
 * and comes back after the last layer, everything between the seven
 * matmuls is a kernel, and each layer's K/V rows come back.)
 *
 * Conventions for every entry point:
 *  - Weights are row-major [out, in] bf16 (passed as uint16_t bit
 *    patterns) and y = x . W^T.  Norm gains are float32 [d].
 *  - Device pointers must be 16-byte aligned.  The library never frees or
 *    keeps a caller pointer past the work it enqueues; all work is ordered
 *    on the caller's stream (a cudaStream_t passed as void*; NULL is the
 *    legacy default stream).
 *  - Errors: every entry point returns a pds_status.  PDS_DECLINED means
 *    the call is not one this library serves, decided on the host before
 *    any device work: nothing was enqueued and no buffer was touched
 *    (cuda_prefill.rs, try_cuda_prefill_dense_stack: None before
 *    touching the device or any cache).  PDS_EINVAL is a bad argument.
 *    PDS_ELAUNCH / PDS_ETIMEOUT are failures after admission: output
 *    buffers and cache rows [start_pos, start_pos+B) may have been
 *    written, rows [0, start_pos) never are; the caller must not advance
 *    its cache length.  The message of the last failure on the calling
 *    thread is pds_last_error(); each distinct failure message is also
 *    printed once per process on stderr (cuda_prefill.rs, warn_once).
 *  - One plan may be used by one stream at a time.
 */
#ifndef PDS_H_
#define PDS_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum pds_status {
  PDS_OK = 0,
  PDS_DECLINED = 1, /* not served; nothing enqueued, nothing touched       */
  PDS_EINVAL = 2,   /* bad pointer, size, alignment or workspace too small */
  PDS_ELAUNCH = 3,  /* a CUDA call failed after admission                  */
  PDS_ETIMEOUT = 4, /* a bounded device-side wait gave up                  */
  PDS_ENOMEM = 5    /* a host or plan-internal device allocation failed    */
} pds_status;

/* RoPE layouts (cuda_prefill.rs, RopeLayoutCuda). */
enum {
  PDS_ROPE_NEOX = 0, /* pair i = channels (i, i + rot_dim/2)  */
  PDS_ROPE_NORM = 1  /* pair i = channels (2i, 2i + 1)        */
};

/*
 * Model dimensions and the run-wide options (cuda_prefill.rs,
 * PrefillParams: n_heads, n_kv_heads, head_dim, rms_eps, attn_softcap,
 * window; LayerRopeCuda: theta, freq_factors, rot_dim, layout, mscale).
 * One rms_eps serves both norms (and the q/k norms); the attention scale
 * is 1/sqrt(head_dim).  Every layer of a run shares the RoPE description,
 * the softcap and the window (a model whose layers differ in them is run as
 * several runs).
 *
 * RoPE: the first rot_dim channels of every q and k head form rot_dim/2
 * pairs (see the layouts); pair i turns by the angle p * omega_i at
 * position p, omega_i = rope_theta^(-2i/rot_dim) / freq_factors[i], and
 * both channels of the pair are multiplied by rope_mscale; channels from
 * rot_dim on pass unchanged.  Softcap: a scaled score z becomes
 * attn_softcap * tanh(z / attn_softcap).  Window: the row at position p
 * sees the keys j with p - window < j <= p.
 *
 * A zero-initialised tail (from rope_layout on) means: Neox over the whole
 * head, no frequency factors, scale 1, no softcap, no window.
 */
typedef struct pds_dims {
  int32_t n_layers;   /* L >= 1                                    */
  int32_t d_model;    /* d: multiple of 128                        */
  int32_t n_heads;    /* H: multiple of n_kv_heads                 */
  int32_t n_kv_heads; /* Hkv                                       */
  int32_t head_dim;   /* hd: 64 or 128; H*hd and Hkv*hd mult. of 128 */
  int32_t ffn_dim;    /* F: multiple of 128                        */
  float rope_theta;   /* > 0                                       */
  float rms_eps;      /* >= 0                                      */
  int32_t rope_layout;        /* PDS_ROPE_NEOX or PDS_ROPE_NORM    */
  int32_t rot_dim;            /* 0 (= head_dim), or a positive multiple of
                                 32 (Neox) / 16 (Norm), <= head_dim */
  const float* freq_factors;  /* host [rot_dim/2] > 0, or NULL (all 1);
                                 copied by pds_plan_create          */
  float rope_mscale;          /* 0 (= 1), or > 0                    */
  float attn_softcap;         /* 0 (none), or > 0                   */
  int32_t window;             /* 0 (none), or > 0 positions         */
} pds_dims;

/*
 * One layer's weights, all device pointers (cuda_prefill.rs,
 * PrefillDenseLayerCuda: attn_norm_w, ffn_norm_w, q, k, v, o, gate, up,
 * down, and the attention extras of AttnExtrasCuda).  The caller owns
 * them; they are read, never written.
 *
 * The extras are optional (NULL: absent), each on its own: a bias is added
 * to its projection's output (after the attention norm's row scale); the
 * q/k norm gains make every head of q / k an RMSNorm of itself,
 * head / sqrt(mean(head^2) + rms_eps) * gain, after the bias and before
 * RoPE.
 */
typedef struct pds_layer {
  const float* attn_norm_w; /* [d]               */
  const float* ffn_norm_w;  /* [d]               */
  const uint16_t* wq;       /* [H*hd,   d]  bf16 */
  const uint16_t* wk;       /* [Hkv*hd, d]  bf16 */
  const uint16_t* wv;       /* [Hkv*hd, d]  bf16 */
  const uint16_t* wo;       /* [d, H*hd]    bf16 */
  const uint16_t* w_gate;   /* [F, d]       bf16 */
  const uint16_t* w_up;     /* [F, d]       bf16 */
  const uint16_t* w_down;   /* [d, F]       bf16 */
  const float* q_bias;      /* [H*hd]   or NULL  */
  const float* k_bias;      /* [Hkv*hd] or NULL  */
  const float* v_bias;      /* [Hkv*hd] or NULL  */
  const float* q_norm;      /* [hd]     or NULL  */
  const float* k_norm;      /* [hd]     or NULL  */
} pds_layer;

typedef struct pds_plan pds_plan;

/*
 * Validate the dimensions and make a plan.
 *
 * Validation is host-only and comes first: PDS_DECLINED (with *out = NULL)
 * for shapes the kernels do not serve (see the field comments of pds_dims)
 * or when the environment variable PDS_DISABLE is set to a non-empty value
 * other than "0" (cuda_prefill.rs: the cuda_dense_enabled() switch), and
 * PDS_EINVAL for a NULL argument or a non-positive size, are decided before
 * any device work.
 *
 * An admitted plan then makes all the device state the library itself
 * allocates, on the device current at this call, which the plan is bound
 * to: a 4-byte status word (cudaMalloc), its 4-byte pinned host copy
 * (cudaMallocHost) and a non-blocking capture stream; PDS_ENOMEM if that
 * fails.  No later call allocates device memory, except that instantiating
 * a CUDA graph of a call (see pds_prefill_dense_stack_device) makes the
 * driver hold memory for its executable graph: at most four per plan, each
 * of 2 + 5 * n_layers kernel nodes, freed by pds_plan_destroy.  Without a
 * CUDA device the plan is host-only: validation and pds_workspace_bytes
 * work, and every call returns PDS_ELAUNCH.
 *
 * Weights are used in place: the kernels read the caller's row-major
 * [out, in] bf16 matrices through TMA tensor maps built at call time
 * (128-byte swizzled boxes straight from the caller's layout), so there is
 * no packing step and no packed copy of the weights.
 */
pds_status pds_plan_create(const pds_dims* dims, pds_plan** out);

/* Release a plan, its device state and its graphs. NULL is a no-op. */
void pds_plan_destroy(pds_plan* plan);

/*
 * Bytes of device workspace for calls with batch <= max_batch and
 * start_pos <= max_start_pos.  The workspace holds the activations between
 * kernels (never the weights or the caches); its content on entry does not
 * matter.  A call needs at least pds_workspace_bytes(plan, batch, 0); what
 * it is given beyond that holds the partial rows of long key ranges, which
 * attention then spreads over all SMs in equal chunks (merged in a fixed
 * order) as far as they fit.  So the schedule, and the rounding of the
 * result, depends on the workspace size: the same inputs with the same
 * workspace size give the same bits.  0 for a NULL plan, max_batch < 1 or
 * max_start_pos < 0.
 */
size_t pds_workspace_bytes(const pds_plan* plan, int32_t max_batch, int32_t max_start_pos);

/*
 * The prefill call, host in / host out (cuda_prefill.rs,
 * try_cuda_prefill_dense_stack and the launch it makes).
 *
 *  layers        host array of n_layers pds_layer (device weight pointers).
 *  k_cache,
 *  v_cache       host arrays of n_layers device pointers, each a bf16 cache
 *                [cache_capacity, n_kv_heads, head_dim].  Rows
 *                [0, start_pos) hold the prefix (K already rotated) and are
 *                only read.  On PDS_OK rows [start_pos, start_pos+batch) hold
 *                this call's new K (post-RoPE) and V rows: these are the
 *                layer's k_rows / v_rows, row b of the batch at row
 *                start_pos+b.
 *  start_pos     s >= 0, the rows already in every cache; new row b is at
 *                position s+b.
 *  batch         B >= 1 new tokens; s+B <= cache_capacity.
 *  hidden_in     host float32 [B, d] (pinned memory makes the copy async
 *                with respect to other host work, pageable also works).
 *  hidden_out    host float32 [B, d]; may alias hidden_in.
 *  workspace     device buffer of >= pds_workspace_bytes(plan, B) bytes.
 *  stream        cudaStream_t as void*.
 *
 * Blocking: returns after the output is in hidden_out (it synchronizes
 * the stream), so device-side timeouts are reported here as PDS_ETIMEOUT.
 */
pds_status pds_prefill_dense_stack(pds_plan* plan, const pds_layer* layers,
                                   uint16_t* const* k_cache, uint16_t* const* v_cache,
                                   int32_t cache_capacity, int32_t start_pos, int32_t batch,
                                   const float* hidden_in, float* hidden_out,
                                   void* workspace, size_t workspace_bytes, void* stream);

/*
 * The same call with device input and output (float32 [B, d] each, may
 * alias), enqueued on the stream without synchronizing.  A device-side
 * timeout is reported by the next pds_plan_sync (or host-I/O call).
 *
 * Launch mode: the first call with a given set of pointers, start_pos and
 * batch captures all of the call's kernels into a CUDA graph, later calls
 * with the same set replay it (four sets are kept per plan, the least
 * recently used is dropped).  A caller whose pointers change on every call
 * can set the environment variable PDS_GRAPH=0 before pds_plan_create to
 * enqueue the kernels one by one instead; the computation is the same.
 */
pds_status pds_prefill_dense_stack_device(pds_plan* plan, const pds_layer* layers,
                                          uint16_t* const* k_cache, uint16_t* const* v_cache,
                                          int32_t cache_capacity, int32_t start_pos,
                                          int32_t batch, const float* hidden_in_dev,
                                          float* hidden_out_dev, void* workspace,
                                          size_t workspace_bytes, void* stream);

/*
 * Synchronize the stream and report whether any bounded device wait of
 * this plan's earlier calls gave up (PDS_ETIMEOUT; the flag is then
 * cleared) or a CUDA error is pending (PDS_ELAUNCH).
 */
pds_status pds_plan_sync(pds_plan* plan, void* stream);

/* Message of the last failure on the calling thread ("" if none). Valid until the next call on that thread. */
const char* pds_last_error(void);

/*
 * Per-kernel timing (measurement support; no counterpart on the pages).
 * While enabled, every kernel of the plan's calls is bracketed by CUDA
 * events recorded on the call's stream, so each kernel's device duration
 * is measured where it runs.  Off by default (events between kernels cost
 * a little).  pds_plan_kernel_times synchronizes the stream, adds the
 * durations of the calls since the last read to the totals and copies the
 * totals out; reset != 0 clears them afterwards.
 */
enum {
  PDS_KERNEL_PREP = 0,   /* RoPE table + first-layer norm prep, once per call */
  PDS_KERNEL_QKV = 1,    /* QKV GEMM + norm scale + RoPE + K/V row write      */
  PDS_KERNEL_ATTN = 2,   /* GQA causal attention                              */
  PDS_KERNEL_WO = 3,     /* wo GEMM + residual + FFN-norm statistics          */
  PDS_KERNEL_GATEUP = 4, /* gate/up GEMM + SwiGLU                             */
  PDS_KERNEL_DOWN = 5,   /* down GEMM + residual + next-norm statistics       */
  PDS_KERNEL_KINDS = 6
};
typedef struct pds_kernel_times {
  int64_t launches[PDS_KERNEL_KINDS];
  double total_ms[PDS_KERNEL_KINDS];
} pds_kernel_times;

/*
 * Failure-detection self test (no counterpart on the pages), a component
 * entry point like the ones below: enqueues on the stream a one-CTA kernel
 * that waits on an mbarrier nothing ever arrives on, through the same
 * bounded wait every tensor-core kernel of the library uses, with a limit of
 * limit_us microseconds (0 < limit_us <= 10 s, else PDS_EINVAL).  The wait
 * gives up, sets the timeout bit of the component status word and the
 * kernel exits; the next pds_component_sync returns PDS_ETIMEOUT.  Returns
 * PDS_OK once enqueued.
 */
pds_status pds_selftest_stuck_wait(uint32_t limit_us, void* stream);

pds_status pds_plan_set_timing(pds_plan* plan, int32_t enable);
pds_status pds_plan_kernel_times(pds_plan* plan, void* stream, pds_kernel_times* out,
                                 int32_t reset);

/*
 * Component entry points: the stack's kernels one at a time, on device
 * buffers, enqueued on the stream (no synchronization).  They serve the
 * kernel-level tests and take the same shape limits as the stack.  Their
 * kernels' bounded waits report a timeout in a status word of the library
 * (one per device), which pds_component_sync reads.
 */

/*
 * Synchronize the stream, then read and clear the component status words
 * of the current device (those of pds_gemm_bf16, pds_gemm_bf16_noalloc,
 * pds_attention and pds_selftest_stuck_wait).  Returns PDS_ETIMEOUT if a
 * bounded device wait of any of their kernels gave up since the previous
 * pds_component_sync on this device (the output of that call is then not
 * valid), PDS_ELAUNCH if the stream reports a CUDA error, else PDS_OK.
 * Allocates nothing.
 */
pds_status pds_component_sync(void* stream);

/*
 * C[M, N] (float32, row-major, ldc = N) = A[M, K] . W[N, K]^T for bf16 A and
 * W (row-major, K contiguous).  M >= 1, N multiple of 128, K multiple of
 * 64.  The same persistent tensor-core GEMM the stack uses, with a plain
 * store epilogue.  `workspace` (device, >= pds_gemm_workspace_bytes(M, N)
 * bytes, 16-byte aligned) holds the partial tiles of the k-split and is
 * written; its content on entry does not matter.
 */
pds_status pds_gemm_bf16(const uint16_t* A, const uint16_t* W, float* C, int32_t M, int32_t N,
                         int32_t K, void* workspace, size_t workspace_bytes, void* stream);

/* Scratch bytes of pds_gemm_bf16 for an M x N output (0 for non-positive sizes). */
size_t pds_gemm_workspace_bytes(int32_t M, int32_t N);

/*
 * pds_gemm_bf16 for callers that cannot allocate device memory: the same
 * product, C[M, N] = A[M, K] . W[N, K]^T, with the same operand rules, but
 * no workspace argument.  The pages have no counterpart; this entry exists
 * for callers that must not call cudaMalloc -- for example a serving
 * process whose device memory is all reserved up front by its own pool,
 * or a plugin that runs inside a host application which owns every
 * allocation -- and so cannot provide the scratch pds_gemm_bf16 takes.
 *
 * The scratch (tile counters and partial tiles of the k-split) lives in a
 * 24 MiB array of the library's own device memory, which every GPU that
 * loads the library holds until the process exits.  Limit: at most 16384
 * output tiles of 128 x 128, i.e. ceil(M/128) * (N/128) <= 16384; larger
 * sizes return PDS_EINVAL with a message and enqueue nothing.  The call
 * allocates nothing (no cudaMalloc, cudaFree or allocating library call).
 *
 * Every call shares the one array and it keeps the last call's contents
 * (the call clears the counters it needs on its stream): calls that overlap
 * on the same GPU, on any streams, race -- order them on one stream or
 * serialize them.  The first call on a device looks up the array's device
 * address for that device (set-up); make that first call before any
 * stream capture.  A device-side timeout of the call is reported by
 * pds_component_sync, which reads and clears the array's status word.
 */
pds_status pds_gemm_bf16_noalloc(const uint16_t* A, const uint16_t* W, float* C, int32_t M,
                                 int32_t N, int32_t K, void* stream);

/*
 * GQA causal attention of B new query rows over a cache (cuda_prefill.rs,
 * PrefillParams: prefix_k/prefix_v, start_pos, attn_scale = 1/sqrt(hd),
 * attn_softcap, window).
 *  q        bf16 [B, H, hd], already rotated (not pre-scaled).
 *  k, v     bf16 [>= start_pos+B, Hkv, hd]; rows [0, start_pos+B) are read.
 *  o        bf16 [B, H*hd]; row b (position p = start_pos + b) attends rows
 *           j <= p, and with window > 0 only p - window < j <= p; query head
 *           h reads kv head h / (H/Hkv).
 *  softcap  0 (none) or > 0: scaled scores z become softcap*tanh(z/softcap).
 *  workspace, workspace_bytes  device scratch for long key ranges (see
 *           pds_attention_workspace_bytes), or NULL and 0.
 * Fails with PDS_DECLINED for hd not in {64, 128} or H % Hkv != 0, and with
 * PDS_EINVAL for a negative softcap or window.
 */
pds_status pds_attention(const uint16_t* q, const uint16_t* k, const uint16_t* v, uint16_t* o,
                         int32_t batch, int32_t start_pos, int32_t n_heads, int32_t n_kv_heads,
                         int32_t head_dim, float softcap, int32_t window, void* workspace,
                         size_t workspace_bytes, void* stream);

/*
 * Workspace bytes with which pds_attention can spread long key ranges over
 * all SMs (its workspace argument; NULL / 0 also works, with long ranges
 * then split over CTA pairs only).  0 for bad sizes.
 */
size_t pds_attention_workspace_bytes(int32_t batch, int32_t start_pos, int32_t n_heads,
                                     int32_t head_dim);

#ifdef __cplusplus
}
#endif

#endif /* PDS_H_ */
