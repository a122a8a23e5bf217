// GQA causal attention of the new rows over the cache prefix plus the new
// rows, on the tcgen05 tensor cores (frink-models 0.29.0
// src/decoder/cuda_prefill.rs, PrefillParams: prefix_k / prefix_v are the
// cache's first start_pos rows; attn_scale = 1/sqrt(head_dim); attn_softcap;
// window).  Query row b sits at position p = start_pos + b, reads kv head
// h / (H / Hkv) and sees keys j <= p (with a window, p - window < j <= p
// only: key tiles wholly below a query tile's windows are not visited).  A
// softcap turns a scaled score z into cap * tanh(z / cap) before the
// softmax.
//
// One CTA per (query head, 128 query rows), heaviest row tiles first.
//   warp 0      TMA producer: the Q tile once, then K and V tiles of 128
//               keys (128-byte swizzle) into two-stage rings, K one ahead
//   warp 1      tcgen05.mma issuer: S_j = Q K_j^T into one of three TMEM
//               buffers, O += P_j V_j into a TMEM accumulator with P_j read
//               from tensor memory (V read MN-major straight from its cache
//               layout); the P.V MMA's completion frees the buffer
//   warps 4-19  softmax, four threads per query row (TMEM lane), each with
//               32 of the tile's keys: S_j from TMEM, causal mask, the row
//               maximum (the quarters exchange theirs through shared
//               memory), exp2 of the scaled score against the row's
//               reference maximum, P_j as bf16 pairs over the first columns
//               of S_j's own buffer.  The reference maximum moves only when
//               a row's maximum grows by more than 2^8 (the O row in TMEM is
//               then rescaled once, after the previous P.V), so exp2 values
//               stay <= 256 and the softmax never otherwise waits for the
//               MMAs: it works on S_{j+1} while O += P_j V_j runs.  At the
//               end the quarters add their row sums in order and each
//               divides and stores a quarter of the O row.
// S_{j+1} is computed while the softmax works on S_j; with three buffers the
// MMA issuer never waits for O += P_{j-1} V_{j-1} to finish before issuing
// S_{j+1}, so the tensor pipe runs S and P.V back to back.
//
// Key-range split: when there are fewer query tiles than SMs, the heaviest
// tiles with long key ranges (as many as fit one CTA per SM) are computed by
// the two CTAs of a cluster, each over half of the tile's key range.  The second CTA sends its
// unnormalised O, row maxima and row sums into the first one's drained
// shared memory (bulk copies), and the first combines the halves in a fixed
// order: O = O0 2^(m0-m) + O1 2^(m1-m) over l0 2^(m0-m) + l1 2^(m1-m).
//
// Every wait is bounded; a wait that gives up sets the status word and the
// CTA exits.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <string>

#include "common.cuh"
#include "fastmath.cuh"
#include "kernels.h"
#include "sm100.cuh"
#include "tc.h"

namespace pds {
namespace {

constexpr int kRows = 128;  // query rows per CTA
constexpr int kKeys = 128;  // keys per tile
constexpr int kRowSplit = 4;  // softmax threads per query row
constexpr int kSoftmaxFirstWarp = 4;
constexpr int kSoftmaxThreads = 128 * kRowSplit;
constexpr int kAttnThreads = 32 * kSoftmaxFirstWarp + kSoftmaxThreads;
constexpr float kRescaleLog2 = 8.0f;  // move the reference max beyond a 2^8 growth
// Shortest key range (in 128-key tiles) worth splitting over a CTA pair: the
// second CTA's prologue and the merge cost about three key tiles (measured:
// splitting 4-tile ranges made the kernel slower, 12.8 -> 14.1 us at 24 heads
// x 512 rows; splitting 15- and 16-tile ranges faster, 26.8 -> 25.2 us).
constexpr int kSplitMinKeyTiles = 8;

template <int HD>
struct AttnCfg {
  static constexpr uint32_t kTile = 128u * HD * 2u;  // Q, K or V tile (bf16)
  // K and V rings: a stage is reloaded only once the MMA that reads it has
  // completed, so a ring of S stages hides a load latency of about S - 1
  // tile times (an L2-resident tile takes ~1.2 us to land)
  static constexpr int kKStages = HD == 128 ? 2 : 3;
  static constexpr int kVStages = 3;
  static constexpr uint32_t kQ = 0;
  static constexpr uint32_t kK0 = kTile;                     // K stage s at kK0 + s kTile
  static constexpr uint32_t kV0 = kK0 + kKStages * kTile;    // V stage s at kV0 + s kTile
  static constexpr uint32_t kP0 = kV0 + kVStages * kTile;    // split: the second half's (l, m)
  static constexpr uint32_t kX = kP0 + 1024u;                // row maxima / sums of the halves
  static constexpr uint32_t kBar = kX + 2u * kRowSplit * 128u * 4u;
  static constexpr int kNumBars = 28;
  static constexpr size_t kSmem = 1024 + kBar + kNumBars * 8 + 16;
  static_assert(kSmem <= 232448, "shared memory per CTA");
  // the split's second half sends its float32 O rows into the K stages
  static_assert(kKStages * kTile >= 128u * HD * 4u, "the O of a split half fits the K stages");
  // TMEM: three S (then P) buffers at columns 0, 128 and 256, O at 384
  static constexpr int kSBufs = 3;
  static constexpr uint32_t kTmO = 384;
  static constexpr uint32_t kTmemCols = 512;
};

struct AttnMaps {
  CUtensorMap q, k, v;
};

// 2^x on the special-function unit (approximate, subnormal results flushed).
__device__ __forceinline__ float exp2_sfu_raw(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
struct AttnArgs {
  uint16_t* o;
  int B, s, H, Hkv;
  float scale_log2;
  uint32_t* status;
  int n_split;  // the first (heaviest) n_split tiles are split over a CTA pair
  float cap_raw;  // softcap over the score scale (raw q.k units); 0: none
  int window;     // 0: none
  // Chunked key ranges (long prefixes): every query tile's key range is cut
  // into ceil(span / chunk) equal chunks, one CTA each, which writes its
  // unnormalised O and its rows' (reference maximum, sum) to o_part /
  // ml_part at its unit; attn_merge_kernel combines them.  0: off.
  int chunk;
  float* o_part;    // [units][128 rows][HD] float32
  float2* ml_part;  // [units][128 rows]
};

// First key tile a query tile starting at position p0 visits: the one that
// holds its first row's first visible key.
__host__ __device__ __forceinline__ int first_key_tile(int p0, int window) {
  return window > 0 ? max(0, p0 - window + 1) / kKeys : 0;
}

// Key tiles [first, first + span) of query tile qt (rows qt*128 ..).
__host__ __device__ __forceinline__ void key_span(int qt, int B, int s, int window, int& first,
                                                  int& span) {
  const int last_row = min((qt + 1) * kRows, B) - 1;
  const int nkt = (s + last_row + 1 + kKeys - 1) / kKeys;
  first = first_key_tile(s + qt * kRows, window);
  span = nkt - first;
}

// Unit u of the chunked mode: query tiles from the last (longest) to the
// first, and within one the chunks, heads fastest.  Sets the query tile,
// head, chunk, chunk count and the chunk's key tiles [kt0, kt0 + n).
__host__ __device__ __forceinline__ bool chunk_unit(int u, int B, int s, int H, int window,
                                                    int chunk, int& qt, int& h, int& c, int& nc,
                                                    int& kt0, int& n) {
  const int nq = (B + kRows - 1) / kRows;
  int base = 0;
  for (qt = nq - 1; qt >= 0; --qt) {
    int first, span;
    key_span(qt, B, s, window, first, span);
    nc = (span + chunk - 1) / chunk;
    if (u < base + nc * H) {
      const int local = u - base;
      c = local / H;
      h = local - c * H;
      kt0 = first + (c * span) / nc;
      n = first + ((c + 1) * span) / nc - kt0;
      return true;
    }
    base += nc * H;
  }
  return false;
}

// c * tanh(x / c) from the identity tanh(y) = 1 - 2 / (e^(2y) + 1), with
// e^(2y) = 2^(x * k2) on the special-function unit (k2 = 2 log2(e) / c);
// it tends to +-c as |x| grows.
__device__ __forceinline__ float softcap_raw(float x, float c, float k2) {
  const float e = exp2_sfu_raw(x * k2);
  return c - __fdividef(2.0f * c, e + 1.0f);
}

// K-major SW128 descriptor of a 128-row operand whose K extent is split in
// 64-element (128-byte) column blocks of 16 KB each.
__device__ __forceinline__ uint64_t kmajor_desc(uint32_t base, int kstep) {
  // k-step of 16 elements: 32 bytes inside a 128-byte block, 4 per block
  return sm100::smem_desc_sw128(base + static_cast<uint32_t>(kstep >> 2) * 16384u +
                                static_cast<uint32_t>(kstep & 3) * 32u);
}

// MN-major SW128 descriptor of the V tile [128 keys][HD] as the B operand
// (N = HD, K = keys) of O += P V: rows are keys (128 bytes of 64 head
// channels each, 8-row groups 1024 bytes apart: the stride byte offset),
// head channels 64..127 are the next 16 KB block (the leading byte offset).
__device__ __forceinline__ uint64_t v_desc(uint32_t base, int kstep) {
  const uint32_t a = base + static_cast<uint32_t>(kstep) * 16u * 128u;  // 16 key rows
  uint64_t d = 0;
  d |= static_cast<uint64_t>((a >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>(16384u >> 4) << 16;  // leading byte offset: next 64 channels
  d |= static_cast<uint64_t>(1024u >> 4) << 32;   // stride byte offset: next 8 keys
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}

__device__ __forceinline__ float exp2_sfu(float x) { return exp2_sfu_raw(x); }

// Pairwise (tree) maximum and sum of n values.
// Maximum of 32 values by three-input maxima (16 instructions).
__device__ __forceinline__ float max32(const float* v) {
  float a[11];
#pragma unroll
  for (int i = 0; i < 10; ++i) a[i] = max3(v[3 * i], v[3 * i + 1], v[3 * i + 2]);
  a[10] = fmaxf(v[30], v[31]);
  const float b0 = max3(a[0], a[1], a[2]), b1 = max3(a[3], a[4], a[5]);
  const float b2 = max3(a[6], a[7], a[8]), b3 = fmaxf(a[9], a[10]);
  return fmaxf(max3(b0, b1, b2), b3);
}
// Sum of 32 values in a fixed pairwise order, two lanes per instruction
// (the values are consumed).
__device__ __forceinline__ float sum32(float* v) {
#pragma unroll
  for (int w = 16; w >= 2; w >>= 1) {
#pragma unroll
    for (int k = 0; k < w / 2; ++k) add2(v[2 * k], v[2 * k + 1], v[2 * k + w], v[2 * k + w + 1]);
  }
  return v[0] + v[1];
}

// kind::f16 instruction descriptor: bf16 x bf16 -> f32, M x N, B MN-major if b_mn.
__host__ __device__ constexpr uint32_t idesc_attn(int M, int N, bool b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (b_mn ? (1u << 16) : 0u) |
         (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

// VAR: the run has a softcap or a window (the plain instantiation carries
// no code for either).
template <int HD, bool VAR>
__global__ void __launch_bounds__(kAttnThreads, 1)
    attn_tc_kernel(const __grid_constant__ AttnMaps maps, const __grid_constant__ AttnArgs a) {
  using namespace sm100;
  using C = AttnCfg<HD>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (sbase - raw);
  const uint32_t bar0 = sbase + C::kBar;
  const uint32_t bar_q = bar0;
  // ring stages (at most 3 of each)
  auto bar_k_full = [&](int st) { return bar0 + 8u * (1 + st); };
  auto bar_k_empty = [&](int st) { return bar0 + 8u * (4 + st); };
  auto bar_v_full = [&](int st) { return bar0 + 8u * (7 + st); };
  auto bar_v_empty = [&](int st) { return bar0 + 8u * (10 + st); };
  // Per TMEM buffer b = j % 3, phase (j / 3) & 1: S_j is in it / it is free
  // again (O += P V of the tile it held has completed) / P_j is in it /
  // O += P_j V_j has completed.  A barrier per buffer keeps every wait within
  // one phase: a softmax warp is at most two tiles ahead of the P.V MMAs.
  auto bar_s_full = [&](int b) { return bar0 + 8u * (13 + b); };
  auto bar_s_free = [&](int b) { return bar0 + 8u * (16 + b); };
  auto bar_p_full = [&](int b) { return bar0 + 8u * (19 + b); };
  auto bar_pv = [&](int b) { return bar0 + 8u * (22 + b); };
  const uint32_t bar_drain = bar0 + 8u * 25;   // every MMA of the CTA has completed
  const uint32_t bar_m_ready = bar0 + 8u * 26;  // split, second CTA: the first may receive
  const uint32_t bar_m_recv = bar0 + 8u * 27;   // split, first CTA: the second's half landed
  uint32_t* misc = reinterpret_cast<uint32_t*>(smem + C::kBar + C::kNumBars * 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // Tiles t = 0, 1, ... run from the longest query tiles to the shortest
  // (head fastest).  With gridDim.x = 2 (clusters of 2 CTAs) cluster c < n_split
  // computes tile c with its key range split in halves, and every later
  // cluster two whole tiles, one per CTA.
  const int nq = (a.B + kRows - 1) / kRows;
  int t = blockIdx.y, half = 0;
  bool split = false;
  if (gridDim.x == 2) {
    half = static_cast<int>(cluster_rank());
    if (t < a.n_split) {
      split = true;
    } else {
      t = a.n_split + 2 * (t - a.n_split) + half;
      half = 0;
      if (t >= a.H * nq) return;
    }
  }
  int qt = nq - 1 - t / a.H;
  int h = t % a.H;
  int kt0, n;  // this CTA's key tiles [kt0, kt0 + n)
  const bool chunked = a.chunk > 0;
  if (chunked) {
    int c, nc;
    if (!chunk_unit(blockIdx.y, a.B, a.s, a.H, VAR ? a.window : 0, a.chunk, qt, h, c, nc, kt0, n))
      return;
  } else {
    const int last_row = min(qt * kRows + kRows, a.B) - 1;
    const int nkt = (a.s + last_row + 1 + kKeys - 1) / kKeys;  // key tiles up to the last row's
    const int kf = VAR ? first_key_tile(a.s + qt * kRows, a.window) : 0;  // first visited
    const int span = nkt - kf;
    const int nk0 = (span + 1) / 2;
    kt0 = kf + ((split && half == 1) ? nk0 : 0);
    n = split ? (half == 0 ? nk0 : span - nk0) : span;
  }
  const int g = h / (a.H / a.Hkv);
  const int b0 = qt * kRows;

  if (threadIdx.x == 0) {
    mbar_init(bar_q, 1);
    for (int i = 0; i < C::kKStages; ++i) {
      mbar_init(bar_k_full(i), 1);
      mbar_init(bar_k_empty(i), 1);
    }
    for (int i = 0; i < C::kVStages; ++i) {
      mbar_init(bar_v_full(i), 1);
      mbar_init(bar_v_empty(i), 1);
    }
    for (int i = 0; i < C::kSBufs; ++i) {
      mbar_init(bar_s_full(i), 1);
      mbar_init(bar_s_free(i), 1);
      mbar_init(bar_p_full(i), kSoftmaxThreads / 32);  // one arrival per softmax warp
      mbar_init(bar_pv(i), 1);
    }
    mbar_init(bar_drain, 1);
    mbar_init(bar_m_ready, 1);
    mbar_init(bar_m_recv, 1);
    *abort_flag = 0;
    mbar_init_fence();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_map(&maps.q);
    tma_prefetch_map(&maps.k);
    tma_prefetch_map(&maps.v);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(misc), C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (split) cluster_sync();  // the peer's barriers are initialised before any remote arrive
  const uint32_t tmem = misc[0];
  grid_dep_launch();

  if (warp == 0) {
    if (lane == 0) {
      // q, k and v are the previous kernel's output
      grid_dep_wait();
      const uint64_t pol = policy_evict_normal();
      mbar_arrive_expect_tx(bar_q, C::kTile);
      for (int c = 0; c < HD / 64; ++c)
        tma_load_2d(sbase + C::kQ + c * 16384u, &maps.q, bar_q, h * HD + c * 64, b0, pol);
      // K_j is freed by S_j, V_j by O += P_j V_j, which comes later.  Each
      // load goes out as soon as its stage is free, K and V independently
      // (neither waits behind the other).
      auto issue = [&](const CUtensorMap* map, uint32_t base, uint32_t full, int st, int j) {
        mbar_arrive_expect_tx(full + 8u * st, C::kTile);
        for (int c = 0; c < HD / 64; ++c)
          tma_load_2d(base + st * C::kTile + c * 16384u, map, full + 8u * st, g * HD + c * 64,
                      (kt0 + j) * kKeys, pol);
      };
      auto stage_free = [&](uint32_t empty, int stages, int j) {
        return j < stages || mbar_try_wait(empty + 8u * (j % stages), ((j / stages) - 1) & 1);
      };
      int kj = 0, vj = 0;
      const uint64_t t0 = global_timer_ns();
      uint32_t idle = 0;
      while (kj < n || vj < n) {
        bool progress = false;
        if (kj < n && stage_free(bar_k_empty(0), C::kKStages, kj)) {
          issue(&maps.k, sbase + C::kK0, bar_k_full(0), kj % C::kKStages, kj);
          ++kj;
          progress = true;
        }
        if (vj < kj && stage_free(bar_v_empty(0), C::kVStages, vj)) {
          issue(&maps.v, sbase + C::kV0, bar_v_full(0), vj % C::kVStages, vj);
          ++vj;
          progress = true;
        }
        // bounded as the mbarrier waits are: give up after their limit, or
        // as soon as another role of the CTA has given up
        if (!progress && (++idle & 63u) == 0) {
          if (*abort_flag) break;
          if (global_timer_ns() - t0 > kWaitLimitNs) {
            *abort_flag = 1;
            atomicOr(a.status, kStatusTimeout);
            break;
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t kIdS = idesc_attn(128, kKeys, false);
      constexpr uint32_t kIdPV = idesc_attn(128, HD, true);
      const uint32_t tm_o = tmem + C::kTmO;
      bool ok = mbar_wait(bar_q, 0, abort_flag, a.status);
      auto issue_s = [&](int j) {
        const int st = j % C::kKStages, sb = j % C::kSBufs;  // K stage, S buffer
        if (!mbar_wait(bar_k_full(st), (j / C::kKStages) & 1, abort_flag, a.status)) return false;
        if (j >= C::kSBufs &&
            !mbar_wait(bar_s_free(sb), ((j / C::kSBufs) - 1) & 1, abort_flag, a.status))
          return false;
        tc_fence_after();
        const uint32_t kb = sbase + C::kK0 + st * C::kTile;
#pragma unroll
        for (int k = 0; k < HD / 16; ++k)
          umma_bf16(tmem + sb * 128u, kmajor_desc(sbase + C::kQ, k), kmajor_desc(kb, k), kIdS,
                    k > 0 ? 1u : 0u);
        umma_commit(bar_s_full(sb));
        umma_commit(bar_k_empty(st));
        return true;
      };
      if (ok) ok = issue_s(0);
      for (int j = 0; ok && j < n; ++j) {
        if (j + 1 < n && !(ok = issue_s(j + 1))) break;
        const int st = j % C::kVStages, sb = j % C::kSBufs;  // V stage, S / P buffer
        if (!(ok = mbar_wait(bar_v_full(st), (j / C::kVStages) & 1, abort_flag, a.status))) break;
        if (!(ok = mbar_wait(bar_p_full(sb), (j / C::kSBufs) & 1, abort_flag, a.status))) break;
        tc_fence_after();
        // P_j (bf16 pairs) sits over the first 64 columns of S_j's buffer
        const uint32_t pt = tmem + sb * 128u;
        const uint32_t vb = sbase + C::kV0 + st * C::kTile;
#pragma unroll
        for (int k = 0; k < kKeys / 16; ++k)
          umma_bf16_ts(tm_o, pt + k * 8u, v_desc(vb, k), kIdPV, (j > 0 || k > 0) ? 1u : 0u);
        umma_commit(bar_v_empty(st));
        umma_commit(bar_pv(sb));
        umma_commit(bar_s_free(sb));
      }
      umma_commit(bar_drain);
      int dummy = 0;
      mbar_wait(bar_drain, 0, &dummy, a.status);
    }
  } else if (warp >= kSoftmaxFirstWarp) {
    const int sw_idx = warp - kSoftmaxFirstWarp;
    const int part = sw_idx >> 2;                           // keys / O columns of this thread
    const int r = (sw_idx & 3) * 32 + lane;                 // query row = TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    float* xch = reinterpret_cast<float*>(smem + C::kX);   // [2 tiles][parts][128 rows]
    constexpr int kPartKeys = kKeys / kRowSplit;
    // the row's position less the first key of this part of key tile 0
    const int rel0 = a.s + b0 + r - (kt0 * kKeys + part * kPartKeys);
    constexpr int kPartCols = HD / kRowSplit;
    static_assert(kPartKeys == 32 && kPartCols % 16 == 0, "TMEM loads and reductions of the parts");
    const float sc = a.scale_log2;
    float m_ref = -INFINITY, l = 0.f;  // m_ref in scaled (base-2) units
    // Every softmax thread passes the named barriers of every tile, even
    // after a wait has given up (ok false: the work is skipped), and a
    // warp's threads agree on ok, so no barrier or warp-wide instruction is
    // left waiting.
    bool ok = true;
    auto wait = [&](uint32_t bar, uint32_t parity) {
      ok = ok && mbar_wait(bar, parity, abort_flag, a.status);
      ok = __all_sync(0xffffffffu, ok);
      if (ok) tc_fence_after();
    };
    // A warp whose 32 rows are all past the batch (a short last query tile,
    // a decode step) keeps every barrier phase of the tile loop, one tile at a
    // time, but computes nothing: the four warps of a lane group share their
    // rows, so they are live or dead together.
    const bool live = b0 + (sw_idx & 3) * 32 < a.B;
    for (int j = 0; j < n; ++j) {
      const int st = j & 1, sb = j % C::kSBufs;  // exchange slot, S / P buffer
      wait(bar_s_full(sb), (j / C::kSBufs) & 1);
      float sv[kPartKeys];
      float mx = -INFINITY;  // raw score maximum (the scale is positive)
      if (ok && !live) {
        // P_j's phase still counts this warp (S_j's wait above keeps it
        // within two tiles of the MMAs, as the live warps are)
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_p_full(sb));
        continue;
      }
      if (ok) {
#pragma unroll
        for (int c = 0; c < kPartKeys / 32; ++c) {
          float t[32];
          tmem_load32(tmem + lane_off + sb * 128u + part * kPartKeys + c * 32, t);
#pragma unroll
          for (int i = 0; i < 32; ++i) sv[c * 32 + i] = t[i];
        }
        // (P_j overwrites S_j's first columns once every part has read its
        // keys: the row maximum's barrier below)
        tc_fence_before();
        if (VAR && a.cap_raw > 0.f) {
          const float k2 = 2.0f * 1.4426950408889634f / a.cap_raw;
#pragma unroll
          for (int i = 0; i < kPartKeys; ++i) sv[i] = softcap_raw(sv[i], a.cap_raw, k2);
        }
        // causal mask (and window) and this part's maximum
        const int rel = rel0 - j * kKeys;  // key i of the part is past the row: i > rel
        if (kPartKeys - 1 > rel - r) {      // some key past some row of the tile
#pragma unroll
          for (int i = 0; i < kPartKeys; ++i)
            if (i > rel) sv[i] = -INFINITY;
        }
        if (VAR && a.window > 0) {  // key i is at or below the window's start: i <= rel - window
          const int lo = rel - a.window;
#pragma unroll
          for (int i = 0; i < kPartKeys; ++i)
            if (i <= lo) sv[i] = -INFINITY;
        }
        mx = max32(sv);
      }
      // the row maximum: all parts
      xch[(st * kRowSplit + part) * 128 + r] = mx;
      named_bar_sync(1 + (warp & 3), 32 * kRowSplit);  // the warps of these 32 rows
      tc_fence_after();
#pragma unroll
      for (int q = 0; q < kRowSplit; ++q) mx = fmaxf(mx, xch[(st * kRowSplit + q) * 128 + r]);
      if (!ok) continue;
      const float mxs = mx * sc;
      float alpha = 1.f;
      bool rescale = false;
      if (j == 0) {
        m_ref = mxs;  // -inf while no key of the CTA's range is visible to the row
      } else if (mxs > m_ref + kRescaleLog2) {  // also from -inf (alpha 0; O and l are 0)
        alpha = exp2f(m_ref - mxs);
        m_ref = mxs;
        rescale = true;
      }
      // P = exp2(s * scale - m_ref) as bf16, and this part's row sum
      uint32_t pk[kPartKeys / 2];
      const float m_use = m_ref == -INFINITY ? 0.f : m_ref;  // masked scores give 0
#pragma unroll
      for (int i = 0; i < kPartKeys / 2; ++i) fma2(sv[2 * i], sv[2 * i + 1], sc, -m_use);
#pragma unroll
      for (int i = 0; i < kPartKeys; ++i) sv[i] = exp2_sfu(sv[i]);
#pragma unroll
      for (int i = 0; i < kPartKeys / 2; ++i) pk[i] = pack_bf16x2(sv[2 * i], sv[2 * i + 1]);
      const float sum = sum32(sv);
      l = l * alpha + sum;
      if (j > 0 && __any_sync(0xffffffffu, rescale)) {
        // O must hold every earlier P V before it is scaled: the last two may
        // still run; they complete in order, so the wait is for the last
        wait(bar_pv((j - 1) % C::kSBufs), ((j - 1) / C::kSBufs) & 1);
        if (!ok) continue;
#pragma unroll
        for (int c = 0; c < kPartCols / 16; ++c) {
          float t[16];
          const uint32_t ta = tmem + lane_off + C::kTmO + part * kPartCols + c * 16;
          tmem_load16(ta, t);
#pragma unroll
          for (int i = 0; i < 16; ++i) t[i] *= alpha;
          tmem_store16(ta, t);
        }
      }
      // P row r, keys of this part: bf16 pairs into columns 16 part .. 16 part
      // + 15 of S_j's buffer (the A operand of O += P_j V_j)
      {
        float pw[kPartKeys / 2];
#pragma unroll
        for (int i = 0; i < kPartKeys / 2; ++i) pw[i] = __uint_as_float(pk[i]);
        tmem_store16_nowait(tmem + lane_off + sb * 128u + part * (kPartKeys / 2), pw);
        tmem_wait_st();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_p_full(sb));
    }
    // the row sum of all parts (in part order), while the last P.V runs;
    // then O row / l
    if (live) {
      named_bar_sync(1 + (warp & 3), 32 * kRowSplit);
      xch[part * 128 + r] = l;
      named_bar_sync(1 + (warp & 3), 32 * kRowSplit);
      l = 0.f;
#pragma unroll
      for (int q = 0; q < kRowSplit; ++q) l += xch[q * 128 + r];
      wait(bar_pv((n - 1) % C::kSBufs), ((n - 1) / C::kSBufs) & 1);
    }
    // split: the second CTA's O part (float32, 16-byte chunks swizzled by the
    // row) goes to the first CTA at the K stages' offset, its row sum and
    // row maximum at the P buffer's offset
    constexpr int kPartChunks = kPartCols / 4;
    const uint32_t o_row = C::kK0 + static_cast<uint32_t>((part * 128 + r) * kPartCols * 4);
    auto o_chunk = [&](int c) {
      return o_row + (static_cast<uint32_t>(c ^ (r & (kPartChunks - 1))) << 4);
    };
    float* lmsg = reinterpret_cast<float*>(smem + C::kP0);  // [128] row sums, then [128] maxima
    if (chunked) {
      // this chunk's unnormalised O row part and the row's (reference max, sum)
      if (ok && live) {
        float* dst = a.o_part + (static_cast<size_t>(blockIdx.y) * kRows + r) * HD + part * kPartCols;
#pragma unroll
        for (int c = 0; c < kPartCols / 16; ++c) {
          float t[16];
          tmem_load16(tmem + lane_off + C::kTmO + part * kPartCols + c * 16, t);
#pragma unroll
          for (int i = 0; i < 4; ++i)
            __stcg(reinterpret_cast<float4*>(dst + c * 16) + i,
                   make_float4(t[4 * i], t[4 * i + 1], t[4 * i + 2], t[4 * i + 3]));
        }
        if (part == 0) __stcg(a.ml_part + static_cast<size_t>(blockIdx.y) * kRows + r,
                              make_float2(m_ref, l));
      }
    } else if (split && half == 1) {
      if (ok && live) {
#pragma unroll
        for (int c = 0; c < kPartCols / 16; ++c) {
          float t[16];
          tmem_load16(tmem + lane_off + C::kTmO + part * kPartCols + c * 16, t);
#pragma unroll
          for (int i = 0; i < 4; ++i)
            *reinterpret_cast<float4*>(smem + o_chunk(4 * c + i)) =
                make_float4(t[4 * i], t[4 * i + 1], t[4 * i + 2], t[4 * i + 3]);
        }
        if (part == 0) {
          lmsg[r] = l;
          lmsg[128 + r] = m_ref;
        }
        fence_proxy_async_smem();
      }
      __syncwarp();
      wait(bar_m_ready, 0);
      if (ok && lane == 0) {
        const uint32_t rbar = mapa_shared(bar_m_recv, 0);
        const uint32_t rows0 = static_cast<uint32_t>((warp & 3) * 32);  // this warp's rows
        const uint32_t o_off = sbase + C::kK0 + (part * 128u + rows0) * kPartCols * 4u;
        bulk_copy_to_cluster(mapa_shared(o_off, 0), o_off, 32u * kPartCols * 4u, rbar);
        if (part == 0) {
          const uint32_t l_off = sbase + C::kP0 + rows0 * 4u;
          bulk_copy_to_cluster(mapa_shared(l_off, 0), l_off, 128u, rbar);
          bulk_copy_to_cluster(mapa_shared(l_off + 512u, 0), l_off + 512u, 128u, rbar);
        }
      }
    } else if (split) {
      if (ok && threadIdx.x == kSoftmaxFirstWarp * 32) {
        mbar_arrive_expect_tx(bar_m_recv, 128u * HD * 4u + 1024u);
        mbar_arrive_cluster(mapa_shared(bar_m_ready, 1));  // O, P and K are done with here
      }
      wait(bar_m_recv, 0);
      if (ok && live) {
        // a row sees its own key, in one half or the other: m is finite (a
        // half that sees none of the row's keys has maximum -inf, weight 0)
        const float m1 = lmsg[128 + r];
        const float m = fmaxf(m_ref, m1);
        const float a0 = m_ref == -INFINITY ? 0.f : exp2f(m_ref - m);
        const float a1 = m1 == -INFINITY ? 0.f : exp2f(m1 - m);
        const float inv = 1.f / (l * a0 + lmsg[r] * a1);
        const int b = b0 + r;
        uint16_t* dst = a.o + (static_cast<size_t>(b) * a.H + h) * HD + part * kPartCols;
#pragma unroll
        for (int c = 0; c < kPartCols / 16; ++c) {
          float t[16];
          tmem_load16(tmem + lane_off + C::kTmO + part * kPartCols + c * 16, t);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float4 o1 = *reinterpret_cast<const float4*>(smem + o_chunk(4 * c + i));
            t[4 * i] = (t[4 * i] * a0 + o1.x * a1) * inv;
            t[4 * i + 1] = (t[4 * i + 1] * a0 + o1.y * a1) * inv;
            t[4 * i + 2] = (t[4 * i + 2] * a0 + o1.z * a1) * inv;
            t[4 * i + 3] = (t[4 * i + 3] * a0 + o1.w * a1) * inv;
          }
          if (b < a.B) {
#pragma unroll
            for (int i = 0; i < 2; ++i)
              reinterpret_cast<uint4*>(dst + c * 16)[i] =
                  make_uint4(pack_bf16x2(t[8 * i], t[8 * i + 1]),
                             pack_bf16x2(t[8 * i + 2], t[8 * i + 3]),
                             pack_bf16x2(t[8 * i + 4], t[8 * i + 5]),
                             pack_bf16x2(t[8 * i + 6], t[8 * i + 7]));
          }
        }
      }
    } else if (ok && live) {
      const float inv = 1.f / l;
      const int b = b0 + r;
      uint16_t* dst = a.o + (static_cast<size_t>(b) * a.H + h) * HD + part * kPartCols;
#pragma unroll
      for (int c = 0; c < kPartCols / 16; ++c) {
        float t[16];
        tmem_load16(tmem + lane_off + C::kTmO + part * kPartCols + c * 16, t);
        if (b < a.B) {
#pragma unroll
          for (int i = 0; i < 2; ++i)
            reinterpret_cast<uint4*>(dst + c * 16)[i] =
                make_uint4(pack_bf16x2(t[8 * i] * inv, t[8 * i + 1] * inv),
                           pack_bf16x2(t[8 * i + 2] * inv, t[8 * i + 3] * inv),
                           pack_bf16x2(t[8 * i + 4] * inv, t[8 * i + 5] * inv),
                           pack_bf16x2(t[8 * i + 6] * inv, t[8 * i + 7] * inv));
        }
      }
    }
  }

  // On a timeout the producer may have copies in flight: let them land.
  if (warp == 0 && lane == 0 && *abort_flag) {
    const uint64_t t0 = global_timer_ns();
    while (global_timer_ns() - t0 < 200000ull) {
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // a split pair: neither CTA leaves while the other may still copy into it
  if (split) cluster_sync();
  if (warp == 1) tmem_dealloc(tmem, C::kTmemCols);
}

// Combines the chunks of the chunked mode: for each query tile, row and
// head, O = sum_c O_c 2^(m_c - m) / sum_c l_c 2^(m_c - m), m = max_c m_c, in
// chunk order.  One warp per (query tile, head, row) -- rows of a tile up to
// the batch (merge_rows) -- lane i holds columns 4i .. 4i + 3.
__host__ __device__ __forceinline__ int merge_rows(int B) { return B < kRows ? B : kRows; }
template <int HD>
__global__ void __launch_bounds__(256) attn_merge_kernel(const __grid_constant__ AttnArgs a) {
  sm100::grid_dep_wait();
  sm100::grid_dep_launch();
  const int warp = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  const int nq = (a.B + kRows - 1) / kRows;
  const int rpt = merge_rows(a.B);
  const int r = warp % rpt;
  int rest = warp / rpt;
  const int h = rest % a.H;
  const int tq = rest / a.H;  // 0: the last query tile (units are ordered that way)
  if (tq >= nq) return;
  const int qt = nq - 1 - tq;
  const int b = qt * kRows + r;
  if (b >= a.B || 4 * lane >= HD) return;
  // the units of this query tile: those of the later (longer) tiles come first
  int base = 0, first = 0, span = 0, nc = 0;
  for (int q = nq - 1; q >= qt; --q) {
    key_span(q, a.B, a.s, a.window, first, span);
    nc = (span + a.chunk - 1) / a.chunk;
    if (q > qt) base += nc * a.H;
  }
  float m = -INFINITY;
  for (int c = 0; c < nc; ++c)
    m = fmaxf(m, a.ml_part[static_cast<size_t>(base + c * a.H + h) * kRows + r].x);
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float l = 0.f;
  for (int c = 0; c < nc; ++c) {
    const size_t u = static_cast<size_t>(base + c * a.H + h);
    const float2 ml = a.ml_part[u * kRows + r];
    if (ml.x == -INFINITY) continue;  // the row sees no key of this chunk
    const float w = exp2f(ml.x - m);
    const float4 o = __ldcg(reinterpret_cast<const float4*>(a.o_part + (u * kRows + r) * HD) + lane);
    acc.x += o.x * w;
    acc.y += o.y * w;
    acc.z += o.z * w;
    acc.w += o.w * w;
    l += ml.y * w;
  }
  const float inv = 1.f / l;
  uint16_t* dst = a.o + (static_cast<size_t>(b) * a.H + h) * HD + 4 * lane;
  *reinterpret_cast<uint2*>(dst) =
      make_uint2(pack_bf16x2(acc.x * inv, acc.y * inv), pack_bf16x2(acc.z * inv, acc.w * inv));
}

// Per-CTA cost beyond its key tiles (prologue, Q load, the partial rows'
// stores), in key-tile times, for the chunk chooser.
constexpr int kChunkOverheadTiles = 3;
// Chunks are at least this many key tiles.
constexpr int kMinChunkTiles = 4;

// Key tiles per chunk for the chunked mode, or 0 when it does not pay: the
// time of a schedule is its waves of resident CTAs times the longest chunk
// plus a CTA's overhead; the chunked mode must beat one CTA per query tile
// by a fifth (the CTA-pair split covers the middle ground).
int choose_chunk(int B, int s, int H, int window, int num_sms, int max_units) {
  const int nq = (B + kRows - 1) / kRows;
  int span_max = 0;
  for (int qt = 0; qt < nq; ++qt) {
    int first, span;
    key_span(qt, B, s, window, first, span);
    span_max = std::max(span_max, span);
  }
  if (num_sms < 1 || max_units < 1) return 0;
  const double waves0 = std::ceil(static_cast<double>(H) * nq / num_sms);
  double best = 0.8 * waves0 * (span_max + kChunkOverheadTiles);
  int best_c = 0;
  for (int c = span_max - 1; c >= kMinChunkTiles; --c) {
    long long units = 0;
    int longest = 0;
    for (int qt = 0; qt < nq; ++qt) {
      int first, span;
      key_span(qt, B, s, window, first, span);
      const int nc = (span + c - 1) / c;
      units += static_cast<long long>(nc) * H;
      longest = std::max(longest, (span + nc - 1) / nc);
    }
    if (units > max_units) break;  // smaller chunks only make more units
    const double cost = std::ceil(static_cast<double>(units) / num_sms) *
                        (longest + kChunkOverheadTiles);
    if (cost < best) {
      best = cost;
      best_c = c;
    }
  }
  return best_c;
}

template <int HD, bool VAR>
pds_status launch_attn_tc(TcContext& c, const uint16_t* q, const uint16_t* k, const uint16_t* v,
                          uint16_t* o, int B, int s, int H, int Hkv, float softcap, int window,
                          cudaStream_t st, std::string* err) {
  using C = AttnCfg<HD>;
  const void* fn = reinterpret_cast<const void*>(attn_tc_kernel<HD, VAR>);
  const cudaError_t attr = kernel_smem_attr(fn, static_cast<int>(C::kSmem));
  if (attr != cudaSuccess) {
    *err = std::string("attention shared-memory attribute: ") + cudaGetErrorString(attr);
    return PDS_ELAUNCH;
  }
  const int T = s + B;
  AttnMaps maps{};
  pds_status rc;
  if ((rc = tc_map_bf16(c, &maps.q, q, static_cast<uint64_t>(H) * HD, B, 128, err)) != PDS_OK)
    return rc;
  if ((rc = tc_map_bf16(c, &maps.k, k, static_cast<uint64_t>(Hkv) * HD, T, 128, err)) != PDS_OK)
    return rc;
  if ((rc = tc_map_bf16(c, &maps.v, v, static_cast<uint64_t>(Hkv) * HD, T, 128, err)) != PDS_OK)
    return rc;
  AttnArgs args{o, B, s, H, Hkv, 1.4426950408889634f / sqrtf(static_cast<float>(HD)), c.status,
                0, softcap > 0.f ? softcap * sqrtf(static_cast<float>(HD)) : 0.f, window,
                0, nullptr, nullptr};
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kAttnThreads);
  cfg.dynamicSmemBytes = C::kSmem;
  cfg.stream = st;
  const int nq = (B + kRows - 1) / kRows, tiles = H * nq;
  // Long key ranges: equal chunks over all SMs, merged by a second kernel.
  const int max_units =
      static_cast<int>(std::min<size_t>(c.attn_ws_bytes / tc_attention_unit_bytes(HD), 1 << 20));
  const int chunk = choose_chunk(B, s, H, VAR ? window : 0, c.num_sms, max_units);
  if (chunk > 0) {
    int units = 0;
    for (int qt = 0; qt < nq; ++qt) {
      int first, span;
      key_span(qt, B, s, VAR ? window : 0, first, span);
      units += H * ((span + chunk - 1) / chunk);
    }
    args.chunk = chunk;
    args.o_part = reinterpret_cast<float*>(c.attn_ws);
    args.ml_part = reinterpret_cast<float2*>(c.attn_ws + static_cast<size_t>(units) * kRows * HD * 4);
    cudaLaunchAttribute at[1];
    int na = 0;
    if (c.pdl) {
      at[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
      at[na].val.programmaticStreamSerializationAllowed = 1;
      ++na;
    }
    cfg.gridDim = dim3(1, units);
    cfg.attrs = at;
    cfg.numAttrs = na;
    cudaError_t ce = cudaLaunchKernelEx(&cfg, attn_tc_kernel<HD, VAR>, maps, args);
    if (ce == cudaSuccess) {
      cudaLaunchConfig_t mc = {};
      mc.gridDim = dim3((tiles * merge_rows(B) + 7) / 8);
      mc.blockDim = dim3(256);
      mc.stream = st;
      mc.attrs = at;
      mc.numAttrs = na;
      ce = cudaLaunchKernelEx(&mc, attn_merge_kernel<HD>, args);
    }
    if (ce != cudaSuccess) {
      *err = std::string("attention launch: ") + cudaGetErrorString(ce);
      return PDS_ELAUNCH;
    }
    return PDS_OK;
  }
  // Split the longest query tiles (a whole row of tiles over the heads at a
  // time) while every CTA still has an SM of its own: fewer tiles than SMs
  // otherwise leave SMs idle behind the longest tiles.
  const int pair_cap = std::min(c.num_sms / 2, kernel_max_clusters(fn, cfg, 2));
  int n_split = 0;
  for (int qt = nq - 1; qt >= 0; --qt) {
    const int nkt = (s + std::min((qt + 1) * kRows, B) + kKeys - 1) / kKeys -
                    first_key_tile(s + qt * kRows, window);
    const int n = n_split + H;
    if (nkt < kSplitMinKeyTiles || n + (tiles - n + 1) / 2 > pair_cap) break;
    n_split = n;
  }
  args.n_split = n_split;
  cudaLaunchAttribute at[2];
  int na = 0;
  if (n_split > 0) {
    cfg.gridDim = dim3(2, n_split + (tiles - n_split + 1) / 2);
    at[na].id = cudaLaunchAttributeClusterDimension;
    at[na].val.clusterDim.x = 2;
    at[na].val.clusterDim.y = 1;
    at[na].val.clusterDim.z = 1;
    ++na;
  } else {
    cfg.gridDim = dim3(1, tiles);
  }
  if (c.pdl) {
    at[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  cfg.attrs = at;
  cfg.numAttrs = na;
  cudaError_t ce = cudaLaunchKernelEx(&cfg, attn_tc_kernel<HD, VAR>, maps, args);
  if (ce != cudaSuccess) {
    *err = std::string("attention launch: ") + cudaGetErrorString(ce);
    return PDS_ELAUNCH;
  }
  return PDS_OK;
}

}  // namespace

size_t tc_attention_unit_bytes(int hd) { return static_cast<size_t>(kRows) * (hd * 4 + 8); }

size_t tc_attention_scratch_bytes(int B, int s, int H, int hd) {
  // the most units the chunked mode can use: chunks of at least
  // kMinChunkTiles key tiles, and no more than 8 per query tile and head
  const int nq = (B + kRows - 1) / kRows;
  long long units = 0;
  for (int qt = 0; qt < nq; ++qt) {
    int first, span;
    key_span(qt, B, s, 0, first, span);
    units += static_cast<long long>(H) * std::min(8, span / kMinChunkTiles);
  }
  return static_cast<size_t>(units) * tc_attention_unit_bytes(hd);
}

pds_status tc_attention(TcContext& c, const uint16_t* q, const uint16_t* k, const uint16_t* v,
                        uint16_t* o, int B, int start_pos, int H, int Hkv, int hd, float softcap,
                        int window, cudaStream_t st, std::string* err) {
  const bool var = softcap > 0.f || window > 0;
  if (hd == 128)
    return var ? launch_attn_tc<128, true>(c, q, k, v, o, B, start_pos, H, Hkv, softcap, window,
                                           st, err)
               : launch_attn_tc<128, false>(c, q, k, v, o, B, start_pos, H, Hkv, 0.f, 0, st, err);
  return var ? launch_attn_tc<64, true>(c, q, k, v, o, B, start_pos, H, Hkv, softcap, window, st,
                                        err)
             : launch_attn_tc<64, false>(c, q, k, v, o, B, start_pos, H, Hkv, 0.f, 0, st, err);
}

}  // namespace pds
