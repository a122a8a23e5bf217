// Persistent tcgen05 GEMM with the stack's fused epilogues.
//
//   C[M, N] = A[M, K] . W[N, K]^T      A, W bf16 (K contiguous), fp32 accumulate
//
// One CTA per SM (384 threads, ~227 KB of shared memory, 2*BN TMEM columns):
//   warp 0      TMA producer: the A box [128 x 64] and the W boxes of each
//               k-block into a ring of S shared-memory stages (128-byte
//               swizzle); weight boxes of the first stages go out before the
//               previous kernel has finished (programmatic dependent launch)
//   warp 1      tcgen05.mma issuer (one thread) into a double-buffered TMEM
//               accumulator; commits free the stages
//   warps 4..11 epilogue: tcgen05.ld of the accumulator (one TMEM lane = one
//               output row; two warps per lane group split the columns),
//               then the fused epilogue (a warp-private shared-memory
//               transpose and row-contiguous stores, or, for a residual
//               GEMM's last tile, shared memory and TMA throughout)
// Warpgroup 0 lowers its registers with setmaxnreg so the epilogue
// warpgroups can hold their fused epilogues without spilling.
//
// CTA pairs: when the row tiles come in pairs, the two CTAs of a cluster
// compute a 256 x BN tile with cta_group::2 MMAs; each loads its own 128
// rows of A and half of the BN weight rows, and the even CTA issues the MMAs.
//
// Work split (grouped stream-K): CTAs form groups of gs (a divisor of the
// row-tile count, up to 8) that take the same (column tile, k-block) ranges
// for different row tiles, so the CTAs reading a weight box run in lockstep
// and the box comes from DRAM once.  The (column tile, k-block) space is cut
// into equal contiguous ranges, one per group.  A tile whose k-blocks are
// spread over several groups is finished by the last CTA to arrive: each
// stores its float32 partial tile to scratch and bumps the tile's counter;
// the one that sees the final count adds the others' partials and its own
// accumulator in k order into its TMEM accumulator (the sum is the same
// whoever arrives last) and runs the epilogue.  No CTA ever waits for
// another.
//
// Cluster split-K (residual GEMMs with few pair tiles): a cluster of 2S CTAs
// computes one 256 x BN tile, pair q over the q-th of S k ranges; the pairs
// exchange column slices of their accumulators through distributed shared
// memory and each finishes its own slice (see split_resid_epilogue).
//
// Row-split cluster (a single row tile of 9..128 rows, any epilogue): a
// cluster of c CTAs (3 to 8) computes one 128 x BN tile, CTA q over the
// q-th of c k ranges; the CTAs exchange row slices of their accumulators
// through distributed shared memory and CTA q finishes rows [q R, q R + R),
// R = 128 / c rounded up to a multiple of 8 (see rsplit_exchange).  Every
// weight byte is read by one CTA, and the weights of a GEMM come in over up
// to eight times as many SMs as it has column tiles, with no partial tile
// in global memory and no CTA reducing the others' partials alone.
//
// Epilogues (the stack's fusions; frink-models 0.29.0
// src/decoder/cuda_prefill.rs, module doc: everything between the seven
// matmuls of a layer is a kernel):
//   plain   store float32 C
//   resid   h = resid + acc; store h; a = bf16(h * gain); per-64-column
//           sum of squares of h (the next RMSNorm's statistics)
//   swiglu  act = silu(r*g) * (r*u): W rows of a tile are 128 gate rows then
//           the same 128 up rows; r = rsqrt(mean sum-of-squares + eps)
//   qkv     r-scaled q|k|v; NeoX RoPE of q and k from a (cos, sin) table;
//           q to the workspace, k and v rows into the caches at start_pos+b
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdlib>
#include <cstdio>
#include <cstring>
#include <map>
#include <mutex>
#include <tuple>
#include <unordered_map>

#include "sm100.cuh"
#include "tc.h"

namespace pds {

namespace {

// Phase hooks for timing studies: a build may define PDS_GEMM_TRACE_HOOK(cta,
// point) to record when each CTA reaches a point; by default they vanish.
#ifndef PDS_GEMM_TRACE_HOOK
#define PDS_GEMM_TRACE_HOOK(cta, point) ((void)0)
#endif

// kEpiQkv is the fast QKV epilogue (Neox over the whole head, no extras);
// kEpiQkvX the general one (biases, q/k head norms, Norm layout, partial
// rotation).
enum EpiKind { kEpiPlain = 0, kEpiResid = 1, kEpiSwiglu = 2, kEpiQkv = 3, kEpiQkvX = 4 };

constexpr int BM = 128;
constexpr int BK = 64;
constexpr int kMinItersPerCta = 4;
// CTAs a GEMM of a single row tile aims for (see make_schedule).
constexpr int kSingleRowCtas = 64;

struct GemmMaps {
  CUtensorMap a;
  CUtensorMap b[3];
  // residual epilogue through shared memory: [0] residual load (float32,
  // 32 x 128 boxes), [1] h store (float32, 32 x 32), [2] a store (bf16, 64 x 32)
  CUtensorMap e[3];
};

struct GemmArgs {
  int M, K;
  int tiles_m, tiles_n, kb;
  // Grouped stream-K schedule: a group is `gs` CTAs that take the same
  // (column tile, k-block) range for `gs` different row tiles, in lockstep,
  // so a weight box comes from DRAM once and is re-read from L2 while hot.
  // A unit is (row-tile group mg < mgs, column tile nt); the units x k-blocks
  // space (`total` iterations) is cut into `groups` equal contiguous ranges.
  int gs, mgs, units, total, groups, grid;
  // Cluster size: 1 (every CTA loads its own tiles), 2 in pair mode, 2*split
  // for the cluster split-K.  No load is shared between CTAs: each CTA's
  // TMA copies fill its own shared memory only.
  int cs;
  // Pair mode (cs = 2): the two CTAs of a cluster compute a 256 x BN tile
  // with cta_group::2 MMAs, each loading its own 128 rows of A and half of
  // the BN weight rows.
  int pair;
  // Cluster split-K (residual GEMMs in pair mode): each cluster of 2*split
  // CTAs computes one 256 x BN tile, pair q over the q-th of `split` equal
  // k ranges, and finishes it through distributed shared memory.  0: off.
  int split;
  // Row-split cluster (a single row tile of more than kSmallRows rows): each
  // cluster of `rsplit` CTAs computes one 128 x BN tile, CTA q over the q-th
  // of rsplit k ranges, and CTA q finishes its slice of rows (see
  // rsplit_exchange).  0: off.
  int rsplit;
  int wrows0, wrows1;  // rows of weight blocks 0 and 1 (concatenated along N)
  int pair_mode;       // W tile = 128 rows of block 0 then the same rows of block 1
  uint32_t* status;
  float* partials;     // [grid][2][BM * BN]
  uint32_t* counters;  // [tiles]
  float* c_out;
  int ldc;
  int resid_n;
  ResidEpilogue resid;
  SwigluEpilogue swiglu;
  QkvEpilogue qkv;
};

// PAIR: the CTA is one of a pair that computes a 256 x BN tile with
// cta_group::2 MMAs; it holds its own 128 rows of A and half of W's BN rows.
template <int BN, bool PAIR = false>
struct Cfg {
  static constexpr int kBRows = PAIR ? BN / 2 : BN;
  static constexpr int kStages = PAIR ? 6 : (BN == 256 ? 4 : 6);
  static constexpr uint32_t kABytes = BM * BK * 2;
  static constexpr uint32_t kBBytes = kBRows * BK * 2;
  static constexpr uint32_t kStage = kABytes + kBBytes;
  static constexpr uint32_t kTmemCols = 2 * BN;
  static constexpr int kBars = 2 * kStages + 5 + 4 + 2;
  // The last tile's residual epilogue reuses the drained stages: 16 KB boxes,
  // BN/32 float32 residual boxes (32 columns x 128 rows) then BN/64 bf16 boxes
  // of the next GEMM's operand (64 columns x 128 rows).
  static constexpr int kBoxesPerStage = static_cast<int>(kStage / 16384);
  static constexpr int kResBoxes = BN / 32;
  static constexpr int kResStages = (kResBoxes + kBoxesPerStage - 1) / kBoxesPerStage;
  // then 4 boxes of other CTAs' partial tiles (2 buffers per column half)
  static constexpr int kPartBoxes = 4;
  static_assert((kResBoxes + kPartBoxes + kBoxesPerStage - 1) / kBoxesPerStage <= kStages,
                "epilogue boxes fit in the stages");
  static_assert(BN * 4 <= 1024, "gain area");
  static_assert(kResStages <= 4, "residual barriers");
  static constexpr uint32_t kMiscBytes = 2048;  // barriers + misc words; the gain from 1024 on
  static constexpr uint32_t kStageBytes = 8 * 32 * 128;         // epilogue staging, 4 KB a warp
  static constexpr size_t kSmem = 1024 + kStages * kStage + kMiscBytes + kStageBytes;
  static_assert(kBars * 8 + 16 <= 1024, "barrier area");

  static_assert(kSmem <= 232448, "shared memory per CTA");
};

// First iteration of group γ's range.
__device__ __forceinline__ int seg_begin(const GemmArgs& g, int grp) {
  return static_cast<int>((static_cast<long long>(grp) * g.total) / g.groups);
}
// The group whose range holds iteration i.
__device__ __forceinline__ int group_of_iter(const GemmArgs& g, int i) {
  return static_cast<int>(((static_cast<long long>(i) + 1) * g.groups - 1) / g.total);
}
// Row and column tile that CTA rank r of a group computes for unit u.
__device__ __forceinline__ void unit_tile(const GemmArgs& g, int u, int r, int& mt, int& nt) {
  nt = u / g.mgs;
  mt = (u - nt * g.mgs) * g.gs + r;
}

struct SegIter {
  int it, end, kb;
  __device__ __forceinline__ bool next(int& tile, int& k0, int& k1) {
    if (it >= end) return false;
    tile = it / kb;
    k0 = it - tile * kb;
    k1 = min(kb, k0 + (end - it));
    it += k1 - k0;
    return true;
  }
};

// Weight block and first row of piece h of column tile nt: the 128-row
// boxes of a tile (BN / 128 of them), or for a CTA pair its half (BN / 2 rows).
template <int BN, bool PAIR>
__device__ __forceinline__ void b_source(const GemmArgs& g, int nt, int h, int& mi, int& row) {
  if (g.pair_mode) {
    mi = h;
    row = nt * 128;
    return;
  }
  const int n0 = nt * BN + h * (PAIR ? BN / 2 : 128);
  if (n0 < g.wrows0) {
    mi = 0;
    row = n0;
  } else if (n0 - g.wrows0 < g.wrows1) {
    mi = 1;
    row = n0 - g.wrows0;
  } else {
    mi = 2;
    row = n0 - g.wrows0 - g.wrows1;
  }
}

// A split tile being finished: contributing groups gf..gl (in k order), this
// CTA's group `me`, rank `r` within the groups, and the unit.
struct Fixup {
  bool active;
  int gf, gl, me, r, unit;
};

// Warpgroup 0: warp 0 is the TMA producer, warp 1 the MMA issuer (and TMEM
// owner), warps 2 and 3 idle.  Epilogue threads: warpgroups 1 and 2 (warps
// 4..11).  Warp w reads TMEM lanes 32*(w%4).. (one output row per thread)
// and takes half of the tile's columns (ch = 0 for warps 4..7, 1 for warps
// 8..11), so two threads share each row.  Warpgroup 0 gives registers to
// the epilogue (setmaxnreg): the launch's 168 per thread become 72 and 216.
constexpr int kEpiWarps = 8;
constexpr int kEpiThreads = 32 * kEpiWarps;
constexpr int kEpiFirstThread = 128;
constexpr int kThreads = kEpiFirstThread + kEpiThreads;
constexpr int kRegsControl = 88;
constexpr int kRegsEpilogue = 208;
static_assert(128 * kRegsControl + kEpiThreads * kRegsEpilogue <= kThreads * 168,
              "register split within the launch's allocation");

// Partial tile of rank r of group grp for unit u: slot 0 if u is the group's
// first unit (its range starts inside u), else slot 1 (u is its last).
__device__ __forceinline__ const float4* partial_slot(const GemmArgs& g, int grp, int r, int u,
                                                      int BN) {
  const int slot = (seg_begin(g, grp) / g.kb == u) ? 0 : 1;
  return reinterpret_cast<const float4*>(g.partials) +
         static_cast<size_t>((grp * g.gs + r) * 2 + slot) * (BM * BN / 4);
}

// Warp-private staging tile of 32 rows x 128 bytes in shared memory, 16-byte
// chunks XOR-swizzled by row, so that a thread-per-row write and a
// four-rows-per-instruction read are both free of bank conflicts.  It turns
// the TMEM layout (one row per thread) into row-contiguous global accesses.
// Two 16-column pieces (chunk ja half ha, chunk jb half hb) of this thread's
// row; without a split the two TMEM loads share one wait.
__device__ __forceinline__ void acc_pair(uint32_t taddr, int ja, int ha, int jb, int hb,
                                         float (&va)[16], float (&vb)[16]) {
  sm100::tmem_load16x2(taddr + ja * 32 + ha * 16, taddr + jb * 32 + hb * 16, va, vb);
}

// x^2 + y^2 + z^2 + w^2 with a fixed rounding order (no contraction), so
// that every epilogue path gives the same statistics bit for bit.
__device__ __forceinline__ float sumsq4(float4 h) {
  return __fadd_rn(__fadd_rn(__fmul_rn(h.x, h.x), __fmul_rn(h.y, h.y)),
                   __fadd_rn(__fmul_rn(h.z, h.z), __fmul_rn(h.w, h.w)));
}

struct Stage {
  float4* base;
  __device__ __forceinline__ float4& at(int row, int q) const { return base[row * 8 + (q ^ (row & 7))]; }
};

// 16 float32 of this thread's row into chunks c..c+3 of its staging row.
__device__ __forceinline__ void stage_f32(const Stage& st, int lane, int c, const float (&v)[16]) {
#pragma unroll
  for (int q = 0; q < 4; ++q)
    st.at(lane, c + q) = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
}

// 16 values of this thread's row as bf16 into chunks c, c+1 of its staging row.
__device__ __forceinline__ void stage_bf16(const Stage& st, int lane, int c, const float (&v)[16]) {
#pragma unroll
  for (int q = 0; q < 2; ++q)
    st.at(lane, c + q) = make_float4(__uint_as_float(pack_bf16x2(v[8 * q], v[8 * q + 1])),
                                     __uint_as_float(pack_bf16x2(v[8 * q + 2], v[8 * q + 3])),
                                     __uint_as_float(pack_bf16x2(v[8 * q + 4], v[8 * q + 5])),
                                     __uint_as_float(pack_bf16x2(v[8 * q + 6], v[8 * q + 7])));
}

// The rows of a warp's 32 that an epilogue stores: lo <= r < hi.
struct Rows {
  int lo, hi;
  __device__ __forceinline__ bool has(int r) const { return r >= lo && r < hi; }
};

// Store staged bf16 chunks c..c+3 (32 columns, 64 bytes) of the warp's rows
// in `rows` to dst_row0 + r * ld, eight rows per instruction.
__device__ __forceinline__ void flush_bf16(const Stage& st, int c, uint16_t* dst_row0, size_t ld,
                                           Rows rows, int lane) {
  // activations are read again soon: keep them in L2 while weights stream by
  const uint64_t pol = sm100::policy_evict_last();
  __syncwarp();
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = i * 8 + (lane >> 2), q = lane & 3;
    if (rows.has(r))
      sm100::st_global_hint(reinterpret_cast<float4*>(dst_row0 + r * ld + q * 8), st.at(r, c + q),
                            pol);
  }
  __syncwarp();
}

// rsqrt(mean of the row's sum-of-squares partials + eps), loads batched.
__device__ __forceinline__ float row_scale(const RowScale& rs, int m) {
  const float* p = rs.ss + static_cast<size_t>(m) * rs.ss_parts;
  float t = 0.f;
#pragma unroll 8
  for (int i = 0; i < rs.ss_parts; ++i) t += p[i];
  return rsqrtf(t * rs.inv_d + rs.eps);
}

// The 32-column chunks of the tile this epilogue thread (column half ch) owns.
template <int BN, int EPI>
__device__ __forceinline__ int owned_chunk(int ch, int i) {
  if constexpr (EPI == kEpiSwiglu) {
    // gate chunks {2ch, 2ch+1} and their up chunks {4+2ch, 5+2ch}
    return (i < 2) ? 2 * ch + i : 4 + 2 * ch + (i - 2);
  } else {
    return ch * (BN / 64) + i;
  }
}
template <int BN, int EPI>
__host__ __device__ constexpr int owned_chunks() {
  return EPI == kEpiSwiglu ? 4 : BN / 64;
}
template <int BN, int EPI>
__device__ __forceinline__ bool chunk_exists(const GemmArgs& g, int nt, int j) {
  if constexpr (EPI == kEpiQkv || EPI == kEpiQkvX)
    return nt * BN + j * 32 < g.qkv.q_width + 2 * g.qkv.kv_width;
  return true;
}

// The (cos, sin) of this thread's row for RoPE channels 0..31, loaded while
// the accumulator is still being made (channels 32..63 of a 128-wide head
// are loaded into the same registers as the first ones are consumed).  The
// table is laid out [channel][row]: one channel's rows are contiguous.
struct RopeRegs {
  float2 v[32];
};
// A (cos, sin) pair through the read-only path, as an opaque load: the
// compiler must keep the value rather than issue the load again at its use.
__device__ __forceinline__ float2 ld_rope(const float2* p) {
  float2 v;
  asm volatile("ld.global.nc.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "l"(p));
  return v;
}
__device__ __forceinline__ const float2* rope_row(const GemmArgs& g, int m) {
  return g.qkv.rope + (m < g.M ? m : 0);
}
template <int BN>
__device__ __forceinline__ void rope_prefetch(const GemmArgs& g, int nt, int ch, int m,
                                              RopeRegs& rr) {
  const QkvEpilogue& e = g.qkv;
  if (nt * BN + ch * 128 >= e.q_width + e.kv_width) return;  // v columns: no rotation
  const float2* cs = rope_row(g, m);
#pragma unroll
  for (int i = 0; i < 32; ++i) rr.v[i] = ld_rope(cs + static_cast<size_t>(i) * e.rope_ld);
}

// 16 floats of a device vector (16-byte aligned: four float4 loads).
__device__ __forceinline__ void ld_f32x16(const float* p, float (&v)[16]) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const float4 t = __ldg(reinterpret_cast<const float4*>(p) + q);
    v[4 * q] = t.x;
    v[4 * q + 1] = t.y;
    v[4 * q + 2] = t.z;
    v[4 * q + 3] = t.w;
  }
}

// The general QKV epilogue of this thread's 128 columns (row `row`, column
// half `ch`): t = r * acc + bias; for q and k every head becomes
// t / sqrt(mean(t^2) + eps) * gain when it has a norm gain, then its first
// rot_dim channels turn in pairs (Neox: (i, i + rot_dim/2); Norm: (2i, 2i+1))
// by the (cos, sin) * mscale of the table; v rows are t.  Values are made
// 16 columns at a time from TMEM (a rotated piece also makes its partner
// piece) and stored through the warp's staging rows, 32 columns at a time.
template <int BN>
__device__ __forceinline__ void qkv_general_epilogue(const GemmArgs& g, uint32_t taddr, int mt,
                                                     int nt, int row, int ch, int lane, float r,
                                                     const Stage& st, Rows rows) {
  const QkvEpilogue& e = g.qkv;
  const int m = mt * BM + row;
  const int m0w = mt * BM + (row & ~31);
  const int c0 = nt * BN + ch * 128;  // first of this thread's 128 columns of [q | k | v]
  if (c0 >= e.q_width + 2 * e.kv_width) return;
  const int blk = c0 < e.q_width ? 0 : (c0 < e.q_width + e.kv_width ? 1 : 2);
  const int cb = c0 - (blk == 0 ? 0 : (blk == 1 ? e.q_width : e.q_width + e.kv_width));
  uint16_t* dst = blk == 0 ? e.q + static_cast<size_t>(m0w) * e.q_width + cb
                           : (blk == 1 ? e.k_cache : e.v_cache) +
                                 static_cast<size_t>(e.start_pos + m0w) * e.kv_width + cb;
  const size_t ld = blk == 0 ? e.q_width : e.kv_width;
  const float* bias = e.bias[blk];
  const uint32_t tcol = taddr + static_cast<uint32_t>(ch * 128);
  // r * acc + bias of columns cc .. cc + 15 (of the 128)
  auto base16 = [&](int cc, float (&v)[16]) {
    sm100::tmem_load16(tcol + cc, v);
#pragma unroll
    for (int k = 0; k < 16; ++k) v[k] *= r;
    if (bias) {
      float b[16];
      ld_f32x16(bias + cb + cc, b);
#pragma unroll
      for (int k = 0; k < 16; ++k) v[k] += b[k];
    }
  };
  auto store32 = [&](int cc, const float (&lo)[16], const float (&hi)[16]) {
    stage_bf16(st, lane, 0, lo);
    stage_bf16(st, lane, 2, hi);
    flush_bf16(st, 0, dst + cc, ld, rows, lane);
  };
  if (blk == 2) {
#pragma unroll 1
    for (int cc = 0; cc < 128; cc += 32) {
      float lo[16], hi[16];
      base16(cc, lo);
      base16(cc + 16, hi);
      store32(cc, lo, hi);
    }
    return;
  }
  const int hd = e.head_dim, R = e.rot_dim, half = R / 2;
  const float* gain = e.norm[blk];
  const float2* cs = rope_row(g, m);
#pragma unroll 1
  for (int hb = 0; hb < 128; hb += hd) {  // heads of these 128 columns
    float scale = 1.f;
    if (gain) {
      float ss = 0.f;
#pragma unroll 1
      for (int cc = hb; cc < hb + hd; cc += 16) {
        float v[16];
        base16(cc, v);
#pragma unroll
        for (int k = 0; k < 16; ++k) ss = fmaf(v[k], v[k], ss);
      }
      scale = rsqrtf(ss / static_cast<float>(hd) + e.rs.eps);
    }
    // channels ic .. ic + 15 of the head, after the head norm
    auto val16 = [&](int ic, float (&v)[16]) {
      base16(hb + ic, v);
      if (gain) {
        float gv[16];
        ld_f32x16(gain + ic, gv);
#pragma unroll
        for (int k = 0; k < 16; ++k) v[k] = v[k] * scale * gv[k];
      }
    };
    // the 16 output channels from ic on
    auto out16 = [&](int ic, float (&o)[16]) {
      if (ic >= R) {
        val16(ic, o);
      } else if (e.rope_layout == PDS_ROPE_NORM) {
        val16(ic, o);
#pragma unroll
        for (int k = 0; k < 16; k += 2) {
          const float2 sc = ld_rope(cs + static_cast<size_t>((ic + k) >> 1) * e.rope_ld);
          const float u = o[k], w = o[k + 1];
          o[k] = u * sc.x - w * sc.y;
          o[k + 1] = u * sc.y + w * sc.x;
        }
      } else {
        const bool first = ic < half;  // the pair's first channel: u cos - w sin
        const int i0 = first ? ic : ic - half;
        float u[16], w[16];
        val16(i0, u);
        val16(i0 + half, w);
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          const float2 sc = ld_rope(cs + static_cast<size_t>(i0 + k) * e.rope_ld);
          o[k] = first ? u[k] * sc.x - w[k] * sc.y : u[k] * sc.y + w[k] * sc.x;
        }
      }
    };
#pragma unroll 1
    for (int ic = 0; ic < hd; ic += 32) {
      float lo[16], hi[16];
      out16(ic, lo);
      out16(ic + 16, hi);
      store32(hb + ic, lo, hi);
    }
  }
}

// The fused epilogue of one tile for this thread (row `row` of the tile,
// column half `ch`); r is the row's RMSNorm scale (SwiGLU and QKV).  The
// warp stores its rows r (of its 32) with wlo <= r < whi that exist.
template <int BN, int EPI>
__device__ __forceinline__ void run_epilogue(const GemmArgs& g, uint32_t taddr, int mt, int nt,
                                             int row, int ch, int lane, float r, const Stage& st,
                                             RopeRegs& rr, int wlo = 0, int whi = 32) {
  const int m = mt * BM + row;
  const int m0w = mt * BM + (row & ~31);                   // first row of this warp's 32
  const Rows rows{wlo, min(whi, g.M - m0w)};               // of which it stores
  if (rows.hi <= rows.lo) return;                          // none: nothing to compute or store
  if constexpr (EPI == kEpiPlain || EPI == kEpiResid) {
    const int q = lane & 7;
    // the residual stream and the next GEMM's operand are read again within
    // the layer: keep them in L2 while the weights stream by
    const uint64_t pol_keep = sm100::policy_evict_last();
    float ss[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) ss[i] = 0.f;
#pragma unroll 1
    for (int c = 0; c < BN / 64; ++c) {
      const int j = ch * (BN / 64) + c;
      const int n0 = nt * BN + j * 32;
      // residual and gain in the row-contiguous layout, in flight before the TMEM reads
      float4 r4[8], g4 = make_float4(1.f, 1.f, 1.f, 1.f);
      if constexpr (EPI == kEpiResid) {
        const ResidEpilogue& e = g.resid;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int rr = i * 4 + (lane >> 3);
          r4[i] = rows.has(rr) ? *reinterpret_cast<const float4*>(
                                  e.resid + static_cast<size_t>(m0w + rr) * g.resid_n + n0 + 4 * q)
                            : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        if (e.gain) g4 = __ldg(reinterpret_cast<const float4*>(e.gain + n0) + q);
      }
      {
        float v0[16], v1[16];
        acc_pair(taddr, j, 0, j, 1, v0, v1);
        stage_f32(st, lane, 0, v0);
        stage_f32(st, lane, 4, v1);
      }
      __syncwarp();
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int rr = i * 4 + (lane >> 3);
        const float4 a4 = st.at(rr, q);
        if constexpr (EPI == kEpiPlain) {
          if (rows.has(rr))
            *reinterpret_cast<float4*>(g.c_out + static_cast<size_t>(m0w + rr) * g.ldc + n0 + 4 * q) = a4;
        } else {
          const ResidEpilogue& e = g.resid;
          const float4 h4 = make_float4(r4[i].x + a4.x, r4[i].y + a4.y, r4[i].z + a4.z, r4[i].w + a4.w);
          const size_t off = static_cast<size_t>(m0w + rr) * g.resid_n + n0 + 4 * q;
          if (rows.has(rr)) sm100::st_global_hint(reinterpret_cast<float4*>(e.out + off), h4, pol_keep);
          if (e.gain) {
            if (rows.has(rr))
              sm100::st_global_hint(
                  reinterpret_cast<uint2*>(e.a_out + off),
                  make_uint2(pack_bf16x2(h4.x * g4.x, h4.y * g4.y), pack_bf16x2(h4.z * g4.z, h4.w * g4.w)),
                  pol_keep);
            float s = sumsq4(h4);
            s += __shfl_xor_sync(0xffffffffu, s, 1);
            s += __shfl_xor_sync(0xffffffffu, s, 2);
            s += __shfl_xor_sync(0xffffffffu, s, 4);
            ss[i] += s;  // the row's sum over this chunk's 32 columns
          }
        }
      }
      __syncwarp();
      if constexpr (EPI == kEpiResid) {
        const ResidEpilogue& e = g.resid;
        if (e.gain && (j & 1)) {  // chunks 2k, 2k+1 make a 64-column group of the statistics
          if (q == 0) {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const int rr = i * 4 + (lane >> 3);
              if (rows.has(rr))
                e.ss_out[static_cast<size_t>(m0w + rr) * (g.resid_n / 64) + (n0 - 32) / 64] = ss[i];
            }
          }
#pragma unroll
          for (int i = 0; i < 8; ++i) ss[i] = 0.f;
        }
      }
    }
  } else if constexpr (EPI == kEpiSwiglu) {
    static_assert(BN == 256, "the SwiGLU tile is 128 gate + 128 up columns");
    const SwigluEpilogue& e = g.swiglu;
#pragma unroll 1
    for (int i = 0; i < 2; ++i) {
      const int jg = 2 * ch + i;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        float gv[16], uv[16];
        acc_pair(taddr, jg, h, 4 + jg, h, gv, uv);
#pragma unroll
        for (int k = 0; k < 16; ++k) gv[k] = silu(r * gv[k]) * (r * uv[k]);
        stage_bf16(st, lane, 2 * h, gv);
      }
      flush_bf16(st, 0, e.act + static_cast<size_t>(m0w) * e.ffn + nt * 128 + jg * 32, e.ffn, rows,
                 lane);
    }
  } else if constexpr (EPI == kEpiQkvX) {
    static_assert(BN == 256, "the QKV tile holds whole heads in each 128-column half");
    qkv_general_epilogue<BN>(g, taddr, mt, nt, row, ch, lane, r, st, rows);
  } else {
    static_assert(BN == 256, "the QKV tile holds whole heads in each 128-column half");
    const QkvEpilogue& e = g.qkv;
    const int c0 = nt * BN + ch * 128;  // this thread's 128 columns of [q | k | v]
    if (c0 >= e.q_width + 2 * e.kv_width) return;
    if (c0 >= e.q_width + e.kv_width) {
      uint16_t* dst = e.v_cache + static_cast<size_t>(e.start_pos + m0w) * e.kv_width +
                      (c0 - e.q_width - e.kv_width);
#pragma unroll 1
      for (int jj = 0; jj < 4; ++jj) {
        float v0[16], v1[16];
        acc_pair(taddr, ch * 4 + jj, 0, ch * 4 + jj, 1, v0, v1);
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          v0[k] *= r;
          v1[k] *= r;
        }
        stage_bf16(st, lane, 0, v0);
        stage_bf16(st, lane, 2, v1);
        flush_bf16(st, 0, dst + jj * 32, e.kv_width, rows, lane);
      }
    } else {
      uint16_t* dst = c0 < e.q_width
                          ? e.q + static_cast<size_t>(m0w) * e.q_width + c0
                          : e.k_cache + static_cast<size_t>(e.start_pos + m0w) * e.kv_width +
                                (c0 - e.q_width);
      const size_t ld = c0 < e.q_width ? e.q_width : e.kv_width;
      // Channels cbase .. cbase + 15 of chunk pair (ja, jb), half h: rotate
      // with the prefetched (cos, sin) and stage both rotated halves.
      auto rotate = [&](int ja, int jb, int h, int cbase) {
        float va[16], vb[16];
        acc_pair(taddr, ch * 4 + ja, h, ch * 4 + jb, h, va, vb);
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          const float2 sc = rr.v[cbase + k];
          const float u = r * va[k], w = r * vb[k];
          va[k] = u * sc.x - w * sc.y;
          vb[k] = u * sc.y + w * sc.x;
        }
        stage_bf16(st, lane, 2 * h, va);
        stage_bf16(st, lane, 4 + 2 * h, vb);
      };
      // head_dim 128: one head per 128 columns; channel i (< 64) pairs with
      // i + 64, i.e. chunk p with chunk p + 2.  head_dim 64: two heads, chunk
      // 2p with chunk 2p + 1.  The rotated halves are staged side by side
      // (chunks 0-3 and 4-7 of the staging row) and stored together.
      if (e.head_dim == 128) {
        // channels 0..31, reloading each 16 with channels 32.. once used
        const float2* cs = rope_row(g, m);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          rotate(0, 2, h, 16 * h);
#pragma unroll
          for (int k = 0; k < 16; ++k)
            rr.v[16 * h + k] = ld_rope(cs + static_cast<size_t>(32 + 16 * h + k) * e.rope_ld);
        }
        flush_bf16(st, 0, dst, ld, rows, lane);
        flush_bf16(st, 4, dst + 2 * 32, ld, rows, lane);
#pragma unroll
        for (int h = 0; h < 2; ++h) rotate(1, 3, h, 16 * h);
        flush_bf16(st, 0, dst + 32, ld, rows, lane);
        flush_bf16(st, 4, dst + 3 * 32, ld, rows, lane);
      } else {
#pragma unroll
        for (int p = 0; p < 2; ++p) {
#pragma unroll
          for (int h = 0; h < 2; ++h) rotate(2 * p, 2 * p + 1, h, 16 * h);
          flush_bf16(st, 0, dst + 2 * p * 32, ld, rows, lane);
          flush_bf16(st, 4, dst + (2 * p + 1) * 32, ld, rows, lane);
        }
      }
    }
  }
}

// A pointer into this CTA's shared memory for a shared-window address, so
// that element accesses are ordinary (reorderable, batchable) C++ loads and
// stores; sm is the dynamic shared memory at window address sbase.
template <typename T>
__device__ __forceinline__ T* sm_at(uint8_t* sm, uint32_t sbase, uint32_t addr) {
  return reinterpret_cast<T*>(sm + (addr - sbase));
}

// Shared-memory address of epilogue box b of a CTA's last tile: the boxes
// fill the stages in the order the ring frees them after the CTA's n_it
// k-blocks, kBoxesPerStage to a stage.
template <int BN, bool PAIR>
__device__ __forceinline__ uint32_t epi_box(uint32_t sbase, int n_it, int b) {
  using C = Cfg<BN, PAIR>;
  const int s = (n_it + b / C::kBoxesPerStage) % C::kStages;
  return sbase + static_cast<uint32_t>(s) * C::kStage +
         static_cast<uint32_t>(b % C::kBoxesPerStage) * 16384u;
}

// Finishes a split tile in TMEM from registers: for each 32-column chunk
// this thread's epilogue reads, the contributors' accumulators are summed
// in k order from zero (its own TMEM value in its place) and written back.
// Two contributors' partial rows are in flight at once.
// Rows past M hold zeros in every contributor (their A rows are zero-filled),
// so their partials are neither stored nor read (row_ok false).
template <int BN, int EPI>
__device__ __forceinline__ void fixup_reduce_regs(const GemmArgs& g, const Fixup& fx,
                                                  uint32_t taddr, int nt, int row, int ch,
                                                  bool row_ok) {
  using namespace sm100;
  constexpr int kOwned = owned_chunks<BN, EPI>();
#pragma unroll 1
  for (int i = 0; i < kOwned; ++i) {
    const int j = owned_chunk<BN, EPI>(ch, i);
    if (!chunk_exists<BN, EPI>(g, nt, j)) continue;
    float v[32];
#pragma unroll
    for (int q = 0; q < 32; ++q) v[q] = 0.f;
#pragma unroll 1
    for (int c0 = fx.gf; c0 <= fx.gl; c0 += 2) {
      float4 b[2][8];
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int c = c0 + u;
        if (c <= fx.gl && c != fx.me && row_ok) {
          const float4* p = partial_slot(g, c, fx.r, fx.unit, BN) + static_cast<size_t>(j * 8) * BM + row;
#pragma unroll
          for (int q = 0; q < 8; ++q) b[u][q] = __ldcg(p + q * BM);
        }
      }
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int c = c0 + u;
        if (c > fx.gl) break;
        if (c == fx.me) {
          float own[32];
          tmem_load32(taddr + j * 32, own);
#pragma unroll
          for (int q = 0; q < 32; ++q) v[q] += own[q];
        } else if (row_ok) {
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            v[4 * q] += b[u][q].x;
            v[4 * q + 1] += b[u][q].y;
            v[4 * q + 2] += b[u][q].z;
            v[4 * q + 3] += b[u][q].w;
          }
        }
      }
    }
    tmem_store32(taddr + j * 32, v);
  }
}

// Split tiles with at most this many rows (decode batches) are finished by
// fixup_reduce_small.
constexpr int kSmallRows = 8;

// Finishes a split tile of at most kSmallRows rows with every epilogue
// thread, in TMEM.  When all contributors' partial rows fit the epilogue
// staging area (`stage`, 32 KB): every thread copies a few of them there
// (all of its loads in flight at once), then every position is summed in k
// order by one thread (this CTA's own partial, stored to its slot like the
// others', in its place) and the rows' owning threads write the sums to
// TMEM.  Otherwise each
// position is summed by one thread, two contributors' loads at a time, and
// the sums reach the owning threads through the staging area.  Called by
// all epilogue threads (et = index).
template <int BN, int EPI>
__device__ __forceinline__ void fixup_reduce_small(const GemmArgs& g, const Fixup& fx,
                                                   uint32_t taddr, int mt, int nt, int row,
                                                   int ch, int et, float4* stage) {
  using namespace sm100;
  const int rv = min(BM, g.M - mt * BM);  // rows of the tile that exist (<= kSmallRows)
  const int per = rv * (BN / 4);          // float4 of one contributor's rows
  const int nc = fx.gl - fx.gf + 1;
  const bool row_ok = row < rv;
  constexpr int kOwned = owned_chunks<BN, EPI>();
  constexpr int kStageF4 = 8 * 32 * 128 / 16;  // float4 in the staging area
  if (nc * per <= kStageF4) {
    const int items = nc * per;
#pragma unroll 1
    for (int b = et; b < items; b += 4 * kEpiThreads) {
      float4 v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int it = b + u * kEpiThreads;
        if (it < items) {
          const int t = it / per, rem = it - t * per;
          const int c4 = rem / rv, rr = rem - c4 * rv;
          v[u] = __ldcg(partial_slot(g, fx.gf + t, fx.r, fx.unit, BN) + static_cast<size_t>(c4) * BM + rr);
        }
      }
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (b + u * kEpiThreads < items) stage[b + u * kEpiThreads] = v[u];
    }
    named_bar_sync(1, kEpiThreads);
    // each position summed in k order by one thread, into contributor 0's place
    for (int pos = et; pos < per; pos += kEpiThreads) {
      float4 acc = stage[pos];
#pragma unroll 1
      for (int t = 1; t < nc; ++t) {
        const float4 x = stage[t * per + pos];
        acc.x += x.x;
        acc.y += x.y;
        acc.z += x.z;
        acc.w += x.w;
      }
      stage[pos] = acc;
    }
    named_bar_sync(1, kEpiThreads);
#pragma unroll 1
    for (int i = 0; i < kOwned; ++i) {
      const int j = owned_chunk<BN, EPI>(ch, i);
      if (!chunk_exists<BN, EPI>(g, nt, j)) continue;
#pragma unroll 1
      for (int h = 0; h < 2; ++h) {
        float v[16];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float4 x = row_ok ? stage[(j * 8 + h * 4 + q) * rv + row]
                                  : make_float4(0.f, 0.f, 0.f, 0.f);
          v[4 * q] = x.x;
          v[4 * q + 1] = x.y;
          v[4 * q + 2] = x.z;
          v[4 * q + 3] = x.w;
        }
        tmem_store16_nowait(taddr + j * 32 + h * 16, v);
      }
    }
    tmem_wait_st();
    named_bar_sync(1, kEpiThreads);  // the staging area is free again
    return;
  }
  float4* sums = stage;  // [BN/4][kSmallRows]
  const int npos = per;
  for (int p = et; p < npos; p += kEpiThreads) {
    const int rr = p % rv, c4 = p / rv;  // row, float4 column (j * 8 + q)
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 1
    for (int c0 = fx.gf; c0 <= fx.gl; c0 += 2) {
      float4 v[2];
#pragma unroll
      for (int u = 0; u < 2; ++u)
        if (c0 + u <= fx.gl)
          v[u] = __ldcg(partial_slot(g, c0 + u, fx.r, fx.unit, BN) + static_cast<size_t>(c4) * BM + rr);
#pragma unroll
      for (int u = 0; u < 2; ++u)
        if (c0 + u <= fx.gl) {
          acc.x += v[u].x;
          acc.y += v[u].y;
          acc.z += v[u].z;
          acc.w += v[u].w;
        }
    }
    sums[c4 * kSmallRows + rr] = acc;
  }
  named_bar_sync(1, kEpiThreads);
#pragma unroll 1
  for (int i = 0; i < kOwned; ++i) {
    const int j = owned_chunk<BN, EPI>(ch, i);
    if (!chunk_exists<BN, EPI>(g, nt, j)) continue;
#pragma unroll 1
    for (int h = 0; h < 2; ++h) {
      float v[16];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float4 x = row_ok ? sums[(j * 8 + h * 4 + q) * kSmallRows + row]
                                : make_float4(0.f, 0.f, 0.f, 0.f);
        v[4 * q] = x.x;
        v[4 * q + 1] = x.y;
        v[4 * q + 2] = x.z;
        v[4 * q + 3] = x.w;
      }
      tmem_store16_nowait(taddr + j * 32 + h * 16, v);
    }
  }
  tmem_wait_st();
  named_bar_sync(1, kEpiThreads);  // the staging area is free again
}

// Finishes a split tile that this CTA completes as its last tile, in TMEM:
// for each 32-column chunk this thread's epilogue reads, the contributors'
// accumulators are summed in k order from zero (its own TMEM value in its
// place), as the register path does, and written back to TMEM.  Every
// thread copies only its own row of the other contributors' partial tiles
// (cp.async, one copy ahead, two buffers per column half in the drained
// stages from box `box0` on), so no thread waits for another.
template <int BN, int EPI, bool PAIR>
__device__ __forceinline__ void fixup_reduce_smem(const GemmArgs& g, const Fixup& fx,
                                                  uint32_t taddr, int nt, int row, int ch,
                                                  uint8_t* sm, uint32_t sbase, int n_it,
                                                  int box0, bool row_ok) {
  using namespace sm100;
  constexpr int kOwned = owned_chunks<BN, EPI>();
  const int nother = fx.gl - fx.gf;  // contributors other than this CTA's group
  // the t-th other contributor in k order, and copy k: (owned chunk, contributor)
  auto contributor = [&](int t) { return fx.gf + t + (fx.gf + t >= fx.me ? 1 : 0); };
  auto issue = [&](int k) {
    const int i = k / nother, t = k - (k / nother) * nother;
    const int j = owned_chunk<BN, EPI>(ch, i);
    const uint32_t dst = epi_box<BN, PAIR>(sbase, n_it, box0 + ch * 2 + (k & 1)) +
                         static_cast<uint32_t>(row) * 16u;
    const float4* src = partial_slot(g, contributor(t), fx.r, fx.unit, BN) +
                        static_cast<size_t>(j * 8) * BM + row;
    if (row_ok) {
#pragma unroll
      for (int q = 0; q < 8; ++q)
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst + q * BM * 16u),
                     "l"(src + q * BM)
                     : "memory");
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
  };
  const int nloads = kOwned * nother;
  issue(0);
  int k = 0;
#pragma unroll 1
  for (int i = 0; i < kOwned; ++i) {
    const int j = owned_chunk<BN, EPI>(ch, i);
    const bool exists = chunk_exists<BN, EPI>(g, nt, j);
    float v[32];
#pragma unroll
    for (int q = 0; q < 32; ++q) v[q] = 0.f;
#pragma unroll 1
    for (int c = fx.gf; c <= fx.gl; ++c) {
      if (c == fx.me) {
        if (exists) {
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            float own[16];
            tmem_load16(taddr + j * 32 + h * 16, own);
#pragma unroll
            for (int q = 0; q < 16; ++q) v[h * 16 + q] += own[q];
          }
        }
        continue;
      }
      if (k + 1 < nloads) {
        issue(k + 1);
        asm volatile("cp.async.wait_group 1;" ::: "memory");
      } else {
        asm volatile("cp.async.wait_group 0;" ::: "memory");
      }
      const uint32_t pb = epi_box<BN, PAIR>(sbase, n_it, box0 + ch * 2 + (k & 1)) +
                          static_cast<uint32_t>(row) * 16u;
      if (row_ok) {
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const float4 p = *sm_at<float4>(sm, sbase, pb + q * BM * 16u);
          v[4 * q] += p.x;
          v[4 * q + 1] += p.y;
          v[4 * q + 2] += p.z;
          v[4 * q + 3] += p.w;
        }
      }
      ++k;
    }
    if (exists) tmem_store32(taddr + j * 32, v);
  }
}

// Residual epilogue of a CTA's last tile, through shared memory, for this
// thread's 32-column chunks jbeg .. jbeg + jcnt - 1 (jbeg even); gain_sm
// holds the tile's BN gains (see resid_gain_prefetch).  The
// producer has loaded the residual boxes of chunks box_base .. into the
// drained stages (box j - box_base, one barrier per stage).  Each thread
// takes its row's accumulator from acc(j, v) (TMEM, or TMEM plus the other
// split contributors' slices), adds it to the residual in place (h), writes
// bf16(h * gain) to its warp's staging area and sums h^2 per 64 columns;
// each warp then stores its 32 rows of each box with TMA.  No global load
// or store of a tile element goes through registers.  The threads of a
// column half (ch) call it together.  Returns false if a wait gave up.
template <int BN, bool PAIR, typename Acc>
__device__ __forceinline__ bool resid_epilogue_smem(const GemmArgs& g, const GemmMaps& maps,
                                                    int mt, int nt, int row, int ch, int lane,
                                                    uint8_t* sm, uint32_t sbase, int n_it,
                                                    uint32_t bar_res0,
                                                    volatile int* abort_flag, const Stage& st,
                                                    float* gain_sm, int jbeg, int jcnt,
                                                    int box_base, Acc&& acc) {
  using namespace sm100;
  using C = Cfg<BN, PAIR>;
  const ResidEpilogue& e = g.resid;
  const int lane_grp = row >> 5;
  const int m = mt * BM + row;
  const int m0w = mt * BM + lane_grp * 32;
  const bool warp_live = m0w < g.M;
  if (!warp_live) return true;  // no row of this warp exists: nothing to compute or store
  const uint64_t pol_keep = policy_evict_last();
  const uint32_t sw = static_cast<uint32_t>(row & 7);
  const uint32_t a_stage = smem_u32(st.base);  // this warp's 32 rows x 64 bf16 of the operand
  // the tile's gain, loaded into shared memory before the accumulator wait
  const float4* gs = reinterpret_cast<const float4*>(gain_sm);
  float ss = 0.f;
#pragma unroll 1
  for (int c = 0; c < jcnt; ++c) {
    const int j = jbeg + c;  // 32-column chunk
    const int b = j - box_base;  // its residual box
    const int n0 = nt * BN + j * 32;
    if (!mbar_wait(bar_res0 + 8u * (b / C::kBoxesPerStage), 0, abort_flag, g.status)) return false;
    float v[32];
    acc(j, v);
    const uint32_t rrow = epi_box<BN, PAIR>(sbase, n_it, b) + static_cast<uint32_t>(row) * 128u;
    if (e.gain && (c & 1) == 0 && c > 0) {
      // the previous pair's operand store has read the staging area
      if (lane == 0) bulk_wait_read_all();
      __syncwarp();
    }
    float t[8];
    float4 rr[8];  // the residual row's 32 columns, all loads in flight at once
#pragma unroll
    for (int q = 0; q < 8; ++q)
      rr[q] = *sm_at<float4>(sm, sbase, rrow + ((static_cast<uint32_t>(q) ^ sw) << 4));
#pragma unroll
    for (int q2 = 0; q2 < 4; ++q2) {
      float4 h[2];
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int q = 2 * q2 + u;
        const float4 r = rr[q];
        h[u] = make_float4(r.x + v[4 * q], r.y + v[4 * q + 1], r.z + v[4 * q + 2],
                           r.w + v[4 * q + 3]);
        *sm_at<float4>(sm, sbase, rrow + ((static_cast<uint32_t>(q) ^ sw) << 4)) = h[u];
        t[q] = sumsq4(h[u]);
      }
      if (e.gain) {
        const float4 ga = gs[j * 8 + 2 * q2], gb = gs[j * 8 + 2 * q2 + 1];
        const uint32_t ac = static_cast<uint32_t>((j & 1) * 4 + q2);
        *sm_at<uint4>(sm, sbase, a_stage + static_cast<uint32_t>(lane) * 128u + ((ac ^ sw) << 4)) =
            make_uint4(pack_bf16x2(h[0].x * ga.x, h[0].y * ga.y),
                       pack_bf16x2(h[0].z * ga.z, h[0].w * ga.w),
                       pack_bf16x2(h[1].x * gb.x, h[1].y * gb.y),
                       pack_bf16x2(h[1].z * gb.z, h[1].w * gb.w));
      }
    }
    // the 32 columns' sum in the register path's shuffle-tree order
    ss += ((t[0] + t[1]) + (t[2] + t[3])) + ((t[4] + t[5]) + (t[6] + t[7]));
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0 && warp_live)
      tma_store_2d(&maps.e[1], epi_box<BN, PAIR>(sbase, n_it, b) + lane_grp * 4096u, n0, m0w,
                   pol_keep);
    if (e.gain && (j & 1)) {
      if (lane == 0 && warp_live) {
        tma_store_2d(&maps.e[2], a_stage, n0 - 32, m0w, pol_keep);
        bulk_commit();
      }
      if (m < g.M) e.ss_out[static_cast<size_t>(m) * (g.resid_n / 64) + (n0 - 32) / 64] = ss;
      ss = 0.f;
    }
  }
  if (lane == 0) {
    bulk_commit();
    bulk_wait_read_all();  // the boxes are read before the CTA's shared memory goes
  }
  __syncwarp();
  return true;
}

// Rows each CTA of a row-split cluster of c finishes: 128 / c rounded up to
// a multiple of 8 (the last slices may be short or empty).
__host__ __device__ __forceinline__ int rsplit_rows(int c) { return ((BM + c - 1) / c + 7) & ~7; }

// Row-split cluster: CTA `me` of the cluster has computed the me-th k range
// of the tile into TMEM and finishes rows [me R, me R + R).
//  1. Once every other CTA of the cluster has said that its stages are free
//     (its accumulator is complete), each warp writes each 32-column chunk
//     of its rows into a shared-memory box of its own (32 rows x 128 bytes,
//     16-byte pieces XOR-swizzled by row) and bulk-copies the rows of each
//     other CTA's slice into that CTA's drained stages, laid out
//     [contributor t][chunk][row of the slice][128 bytes].  The received
//     slices and the outgoing boxes share the drained stages, none reused.
//  2. Once its own slices have landed, all epilogue threads fold them, each
//     16-byte piece of the slice by one thread, into the sum of the ranks
//     before this CTA's and the sum of those after it (each in rank order,
//     from zero), written over contributor slots 0 and c - 2.
//  3. The warps that hold the slice's rows in TMEM make (before + own) +
//     after and write it back to TMEM for the epilogue.
// The order of the additions is fixed, so the result does not depend on
// timing.  Every epilogue thread reaches the barrier between 2 and 3, and
// all leave on the abort flag after it, so a wait that gives up cannot
// split the CTA.  Returns false if a wait gave up.
template <int BN, int EPI>
__device__ __forceinline__ bool rsplit_exchange(const GemmArgs& g, uint32_t taddr, int row, int ch,
                                                int lane, uint8_t* sm, uint32_t sbase,
                                                uint32_t bar_ready, uint32_t bar_recv,
                                                volatile int* abort_flag, int me, bool leader) {
  using namespace sm100;
  constexpr int kOwned = owned_chunks<BN, EPI>();
  constexpr int kChunks = BN / 32;
  const int c = g.rsplit, R = rsplit_rows(c);
  const int lo = me * R, hs = lo + R, hi = min(g.M, hs);  // the rows this CTA finishes
  const int n = max(0, hi - lo);
  auto recv_off = [&](int t, int j, int r) {
    return static_cast<uint32_t>(((t * kChunks + j) * R + r) * 128);
  };
  const uint32_t slot_bytes = static_cast<uint32_t>(kChunks * R * 128);  // one contributor's
  const uint32_t recv_bytes = static_cast<uint32_t>(c - 1) * slot_bytes;
  if (leader) {
    mbar_arrive_expect_tx(bar_recv, static_cast<uint32_t>((c - 1) * n * BN * 4));
    for (int p = 0; p < c; ++p)
      if (p != me) mbar_arrive_cluster(mapa_shared(bar_ready, static_cast<uint32_t>(p)));
  }
  bool ok = __all_sync(0xffffffffu, mbar_wait(bar_ready, 0, abort_flag, g.status));
  const int w0 = row & ~31, lg = w0 / 32;  // this warp's rows w0 .. w0 + 31
  const uint32_t sw = static_cast<uint32_t>(row & 7);
  if (ok) {
    tc_fence_after();
    // lane group l holds rows of other slices that exist
    auto sends_of = [&](int l) {
      return 32 * l < g.M && (32 * l < lo || min(32 * l + 32, g.M) > hs);
    };
    // this warp's boxes: a slot per lane group that sends, two halves each
    int slot = 0;
    for (int l = 0; l < lg; ++l) slot += sends_of(l) ? 1 : 0;
    if (sends_of(lg)) {
#pragma unroll 1
      for (int k = 0; k < kOwned; ++k) {
        const int j = owned_chunk<BN, EPI>(ch, k);
        const uint32_t box =
            sbase + recv_bytes + static_cast<uint32_t>(((slot * 2 + ch) * kOwned + k) * 4096);
        float v[32];
        tmem_load32(taddr + j * 32, v);
        const uint32_t mine_row = box + static_cast<uint32_t>(lane) * 128u;
#pragma unroll
        for (int q4 = 0; q4 < 8; ++q4)
          *sm_at<float4>(sm, sbase, mine_row + ((static_cast<uint32_t>(q4) ^ sw) << 4)) =
              make_float4(v[4 * q4], v[4 * q4 + 1], v[4 * q4 + 2], v[4 * q4 + 3]);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          // the existing rows of each other CTA's slice among this warp's
          for (int p = w0 / R; p < c && p * R < w0 + 32; ++p) {
            if (p == me) continue;
            const int a = max(w0, p * R), b = min(min(w0 + 32, p * R + R), g.M);
            if (a >= b) continue;
            const int t = me < p ? me : me - 1;
            bulk_copy_to_cluster(
                mapa_shared(sbase + recv_off(t, j, a - p * R), static_cast<uint32_t>(p)),
                box + static_cast<uint32_t>(a - w0) * 128u, static_cast<uint32_t>(b - a) * 128u,
                mapa_shared(bar_recv, static_cast<uint32_t>(p)));
          }
        }
      }
    }
    ok = __all_sync(0xffffffffu, mbar_wait(bar_recv, 0, abort_flag, g.status));
  }
  // 2. before / after sums of the received slices, one 16-byte piece a thread
  const uint32_t before = sbase, after = sbase + static_cast<uint32_t>(me > 0 ? c - 2 : 0) * slot_bytes;
  if (ok) {
    const int et = static_cast<int>(threadIdx.x) - kEpiFirstThread;
#pragma unroll 1
    for (int idx = et; idx < kChunks * n * 8; idx += kEpiThreads) {
      const int q4 = idx & 7, rest = idx >> 3, r = rest % n, j = rest / n;
      const uint32_t off = recv_off(0, j, r) + ((static_cast<uint32_t>(q4) ^ (r & 7)) << 4);
      // all contributors' pieces in flight at once (c - 1 <= 7), then the
      // two sums in rank order
      float4 x[7];
#pragma unroll
      for (int t = 0; t < 7; ++t)
        if (t < c - 1) x[t] = *sm_at<float4>(sm, sbase, sbase + static_cast<uint32_t>(t) * slot_bytes + off);
      float4 pre = make_float4(0.f, 0.f, 0.f, 0.f), post = pre;
#pragma unroll
      for (int t = 0; t < 7; ++t) {
        if (t < me) {
          pre.x += x[t].x;
          pre.y += x[t].y;
          pre.z += x[t].z;
          pre.w += x[t].w;
        } else if (t < c - 1) {
          post.x += x[t].x;
          post.y += x[t].y;
          post.z += x[t].z;
          post.w += x[t].w;
        }
      }
      if (me > 0) *sm_at<float4>(sm, sbase, before + off) = pre;
      if (me < c - 1) *sm_at<float4>(sm, sbase, after + off) = post;
    }
  }
  named_bar_sync(1, kEpiThreads);
  if (*abort_flag) return false;
  // 3. (before + own) + after, by the warps that hold the slice's rows
  if (n == 0 || w0 >= hi || w0 + 32 <= lo) return true;
  const bool mine = row >= lo && row < hi;
  const int r = mine ? row - lo : 0;
#pragma unroll 1
  for (int i = 0; i < kOwned; ++i) {
    const int j = owned_chunk<BN, EPI>(ch, i);
    float own[32];
    tmem_load32(taddr + j * 32, own);
    if (mine) {
      const uint32_t roff = recv_off(0, j, r);
      if (me > 0) {
#pragma unroll
        for (int q4 = 0; q4 < 8; ++q4) {
          const float4 x =
              *sm_at<float4>(sm, sbase, before + roff + ((static_cast<uint32_t>(q4) ^ sw) << 4));
          own[4 * q4] = x.x + own[4 * q4];
          own[4 * q4 + 1] = x.y + own[4 * q4 + 1];
          own[4 * q4 + 2] = x.z + own[4 * q4 + 2];
          own[4 * q4 + 3] = x.w + own[4 * q4 + 3];
        }
      }
      if (me < c - 1) {
#pragma unroll
        for (int q4 = 0; q4 < 8; ++q4) {
          const float4 x =
              *sm_at<float4>(sm, sbase, after + roff + ((static_cast<uint32_t>(q4) ^ sw) << 4));
          own[4 * q4] += x.x;
          own[4 * q4 + 1] += x.y;
          own[4 * q4 + 2] += x.z;
          own[4 * q4 + 3] += x.w;
        }
      }
    }
    tmem_store16_nowait(taddr + j * 32, reinterpret_cast<const float(&)[16]>(own[0]));
    tmem_store16_nowait(taddr + j * 32 + 16, reinterpret_cast<const float(&)[16]>(own[16]));
  }
  tmem_wait_st();
  return true;
}

// The gains of the BN columns of column tile nt into shared memory, by the
// epilogue threads, before they wait for the CTA's last accumulator (the
// gain is a weight: it does not wait for the previous kernel).
template <int BN>
__device__ __forceinline__ void resid_gain_prefetch(const GemmArgs& g, int nt, float* gain_sm,
                                                    int et) {
  if (g.resid.gain && et < BN / 4)
    reinterpret_cast<float4*>(gain_sm)[et] =
        __ldg(reinterpret_cast<const float4*>(g.resid.gain + nt * BN) + et);
  sm100::named_bar_sync(1, kEpiThreads);
}

// Cluster split-K of a residual GEMM: the cluster's S pairs compute one
// 256 x BN tile over S consecutive k ranges.  The tile's eight 32-column
// chunks are dealt to the pairs in 64-column units (pair q finishes chunks
// [first, first + count)); every CTA sends the chunks it does not finish
// to the CTA of the same rank in the finishing pair, straight into that
// CTA's drained stages (after its residual boxes), and finishes its own.
struct SplitSlice {
  int first, count;
};
__host__ __device__ __forceinline__ SplitSlice split_slice(int S, int q) {
  const int base = 4 / S, extra = 4 % S;
  const int units = base + (q < extra ? 1 : 0);
  const int first = q * base + (q < extra ? q : extra);
  return SplitSlice{2 * first, 2 * units};
}
__device__ __forceinline__ int split_owner(int S, int j) {
  for (int q = 0; q < S - 1; ++q) {
    const SplitSlice sl = split_slice(S, q);
    if (j < sl.first + sl.count) return q;
  }
  return S - 1;
}
// Box of the finishing CTA (pair q, slice sl) that receives chunk j from pair p.
__device__ __forceinline__ int split_recv_box(int S, int q, const SplitSlice& sl, int j, int p) {
  return sl.count + (j - sl.first) * (S - 1) + (p < q ? p : p - 1);
}

// The split epilogue of one CTA (pair p of the cluster, rank r in the
// pair).  Returns false if a wait gave up.
template <int BN>
__device__ __forceinline__ bool split_resid_epilogue(
    const GemmArgs& g, const GemmMaps& maps, uint32_t taddr, int mt, int nt, int row, int ch,
    int lane, uint8_t* sm, uint32_t sbase, int grp, uint32_t bar_res0, uint32_t bar_ready,
    uint32_t bar_recv,
    volatile int* abort_flag, const Stage& st, float* gain_sm, uint32_t crank, bool leader) {
  using namespace sm100;
  static_assert(BN == 256, "eight 32-column chunks in four 64-column units");
  constexpr bool PAIR = true;
  const int S = g.split;
  const int p = static_cast<int>(crank >> 1), r = static_cast<int>(crank & 1u);
  const int grp0 = grp - p;  // the cluster's first group
  auto n_it_of = [&](int q) { return seg_begin(g, grp0 + q + 1) - seg_begin(g, grp0 + q); };
  const SplitSlice mine = split_slice(S, p);
  const int my_n_it = n_it_of(p);
  // 1. receive: expect the other pairs' slices, then tell them our stages
  //    are free (every MMA of this pair has completed: the accumulator is full)
  if (leader) {
    mbar_arrive_expect_tx(bar_recv, static_cast<uint32_t>(mine.count * (S - 1)) * 16384u);
    for (int q = 0; q < S; ++q)
      if (q != p) mbar_arrive_cluster(mapa_shared(bar_ready, static_cast<uint32_t>(2 * q + r)));
  }
  // 2. send: this half's share of the chunks other pairs finish.  With room
  //    in the drained stages after the received slices, a chunk is staged
  //    there and each warp bulk-copies its 32 rows (4 KB); otherwise the
  //    rows go out as 16-byte asynchronous remote stores.
  if (!mbar_wait(bar_ready, 0, abort_flag, g.status)) return false;
  tc_fence_after();
  {
    const int out_box0 = mine.count * S;  // first free box of the drained stages
    const bool bulk = out_box0 + (BN / 32 - mine.count) <= Cfg<BN, PAIR>::kStages * 2;
    const uint32_t sw = static_cast<uint32_t>(row & 7);
    const uint32_t wrow0 = static_cast<uint32_t>(row & ~31) * 128u;  // this warp's 32 rows
    int k = 0;
#pragma unroll 1
    for (int j = 0; j < BN / 32; ++j) {
      if (j >= mine.first && j < mine.first + mine.count) continue;
      const int kk = k++;
      if ((kk & 1) != ch) continue;
      const int q = split_owner(S, j);
      const SplitSlice sl = split_slice(S, q);
      const uint32_t dst_rank = static_cast<uint32_t>(2 * q + r);
      const uint32_t dst_box = epi_box<BN, PAIR>(sbase, n_it_of(q), split_recv_box(S, q, sl, j, p));
      const uint32_t rbar = mapa_shared(bar_recv, dst_rank);
      float v[32];
      tmem_load32(taddr + j * 32, v);
      if (bulk) {
        const uint32_t src_box = epi_box<BN, PAIR>(sbase, my_n_it, out_box0 + kk);
        const uint32_t src = src_box + static_cast<uint32_t>(row) * 128u;
#pragma unroll
        for (int q4 = 0; q4 < 8; ++q4)
          *sm_at<float4>(sm, sbase, src + ((static_cast<uint32_t>(q4) ^ sw) << 4)) =
              make_float4(v[4 * q4], v[4 * q4 + 1], v[4 * q4 + 2], v[4 * q4 + 3]);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0)
          bulk_copy_to_cluster(mapa_shared(dst_box + wrow0, dst_rank), src_box + wrow0, 4096u,
                               rbar);
      } else {
        const uint32_t dst = mapa_shared(dst_box + static_cast<uint32_t>(row) * 128u, dst_rank);
#pragma unroll
        for (int q4 = 0; q4 < 8; ++q4)
          st_async_f4(dst + ((static_cast<uint32_t>(q4) ^ sw) << 4),
                      make_float4(v[4 * q4], v[4 * q4 + 1], v[4 * q4 + 2], v[4 * q4 + 3]), rbar);
      }
    }
  }
  // 3. finish this pair's chunks: the contributors in k order (pair order)
  if (!mbar_wait(bar_recv, 0, abort_flag, g.status)) return false;
  auto acc = [&](int j, float (&v)[32]) {
    float own[32];
    tmem_load32(taddr + j * 32, own);
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = 0.f;
    const uint32_t sw = static_cast<uint32_t>(row & 7);
    for (int q = 0; q < S; ++q) {
      if (q == p) {
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] += own[i];
      } else {
        const uint32_t src = epi_box<BN, PAIR>(sbase, my_n_it, split_recv_box(S, p, mine, j, q)) +
                             static_cast<uint32_t>(row) * 128u;
#pragma unroll
        for (int q4 = 0; q4 < 8; ++q4) {
          const float4 x = *sm_at<float4>(sm, sbase, src + ((static_cast<uint32_t>(q4) ^ sw) << 4));
          v[4 * q4] += x.x;
          v[4 * q4 + 1] += x.y;
          v[4 * q4 + 2] += x.z;
          v[4 * q4 + 3] += x.w;
        }
      }
    }
  };
  // halves: two 64-column units each, or the first half alone for one unit
  const int half_cnt = mine.count >= 4 ? mine.count / 2 : (ch == 0 ? mine.count : 0);
  const int jbeg = mine.first + (mine.count >= 4 ? ch * (mine.count / 2) : 0);
  if (half_cnt == 0) return true;
  return resid_epilogue_smem<BN, PAIR>(g, maps, mt, nt, row, ch, lane, sm, sbase, my_n_it,
                                       bar_res0, abort_flag, st, gain_sm, jbeg, half_cnt,
                                       mine.first, acc);
}

// RSPLIT: the row-split cluster schedule (g.rsplit > 1; non-pair only), a
// separate instantiation so that neither schedule's registers burden the other.
template <int BN, int EPI, bool PAIR, bool RSPLIT>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_kernel(const __grid_constant__ GemmMaps maps, const __grid_constant__ GemmArgs g) {
  static_assert(!(PAIR && RSPLIT), "a row-split cluster computes single row tiles");
  using namespace sm100;
  using C = Cfg<BN, PAIR>;
  constexpr int S = C::kStages;
  constexpr uint32_t kIdesc = idesc_bf16_f32(PAIR ? 2 * BM : BM, BN);

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (sbase - raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S * C::kStage);
  uint32_t* misc = reinterpret_cast<uint32_t*>(bars + C::kBars);  // [0] tmem base [1] count [2] abort
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 2);
  const uint32_t bar0 = smem_u32(bars);
  auto bar_full = [&](int s) { return bar0 + 8u * s; };
  auto bar_empty = [&](int s) { return bar0 + 8u * (S + s); };
  auto bar_tfull = [&](int a) { return bar0 + 8u * (2 * S + a); };
  auto bar_tempty = [&](int a) { return bar0 + 8u * (2 * S + 2 + a); };
  const uint32_t bar_drain = bar0 + 8u * (2 * S + 4);
  const uint32_t bar_res0 = bar0 + 8u * (2 * S + 5);  // residual boxes landed, one per stage
  const uint32_t bar_ready = bar0 + 8u * (2 * S + 9);  // split: the other pairs may send
  const uint32_t bar_recv = bar0 + 8u * (2 * S + 10);  // split: their slices have landed

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cta = blockIdx.x;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(bar_full(s), 1);
      // freed by this CTA's MMAs, or for a pair by the even CTA's
      mbar_init(bar_empty(s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(bar_tfull(a), 1);
      // one arrival per epilogue warp (of both CTAs of a pair)
      mbar_init(bar_tempty(a), PAIR ? 2 * kEpiWarps : kEpiWarps);
    }
    mbar_init(bar_drain, 1);
    for (int f = 0; f < 4; ++f) mbar_init(bar_res0 + 8u * f, 1);
    mbar_init(bar_ready, g.split > 1 ? g.split - 1 : (RSPLIT ? g.rsplit - 1 : 1));
    mbar_init(bar_recv, 1);
    *abort_flag = 0;
    mbar_init_fence();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_map(&maps.a);
    tma_prefetch_map(&maps.b[0]);
    tma_prefetch_map(&maps.b[1]);
    tma_prefetch_map(&maps.b[2]);
    if (EPI == kEpiResid) {
      tma_prefetch_map(&maps.e[0]);
      tma_prefetch_map(&maps.e[1]);
      tma_prefetch_map(&maps.e[2]);
    }
  }
  if (warp == 1) {
    if constexpr (PAIR) {
      tmem_alloc_pair(smem_u32(misc), C::kTmemCols);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(smem_u32(misc), C::kTmemCols);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // the peers of a pair or split cluster arrive on this CTA's barriers
  if (g.cs > 1) cluster_sync();
  const uint32_t tmem_base = misc[0];
  // A pair (cluster ranks 2k, 2k+1): the even CTA issues the MMAs and owns
  // the stage-full and accumulator-empty barriers both CTAs' copies and
  // epilogues signal.
  const uint32_t crank = g.cs > 1 ? cluster_rank() : 0u;
  const uint32_t prank = PAIR ? (crank & 1u) : 0u;
  const uint32_t lead = crank & ~1u;  // the pair leader's cluster rank
  const uint16_t pmask = static_cast<uint16_t>(3u << lead);
  if (threadIdx.x == 0) PDS_GEMM_TRACE_HOOK(cta, 0);

  // Everything above overlaps the previous kernel when launched with
  // programmatic stream serialization.  Only the activations (A), the
  // epilogue's inputs and its outputs depend on that kernel: the producer
  // starts the weight loads of its first stages before waiting for it, the
  // epilogue warps wait before they touch global memory, and the MMA warp
  // only sees shared memory and TMEM.
  grid_dep_launch();

  const int grp = cta / g.gs, rank = cta - grp * g.gs;
  const int it0 = seg_begin(g, grp), it1 = seg_begin(g, grp + 1);
  int issued = 0;  // producer: k-block loads issued
  int consumed = 0;

  // Each role changes its registers first thing, so that its code is
  // compiled for its own register count (warps 0..3 lower theirs, the
  // epilogue warpgroups take them).
  if (warp == 0) {
    setmaxnreg_dec<kRegsControl>();
    if (lane == 0) {
      // A (activations) is re-read by every column tile: keep it.  A weight
      // box is read once when one cluster (or CTA) holds all the row tiles of
      // its group, or in a row-split cluster (one CTA per k range): let it
      // go first; otherwise the group's other CTAs read it again right away:
      // normal priority.
      const uint64_t pol_a = policy_evict_last();
      const uint64_t pol_w =
          (g.cs == g.gs || RSPLIT) ? policy_evict_first() : policy_evict_normal();
      // where a stage's copies complete: the pair leader's barrier, or our own
      auto full_bar = [&](int s) { return PAIR ? mapa_shared(bar_full(s), lead) : bar_full(s); };
      auto load_w = [&](int s, int nt, int kb) {
        if constexpr (PAIR) {
          // this CTA's half of the pair's BN weight rows
          int mi, row;
          b_source<BN, true>(g, nt, static_cast<int>(prank), mi, row);
          tma_load_2d_pair(sbase + s * C::kStage + C::kABytes, &maps.b[mi], full_bar(s), kb * BK,
                           row, pol_w);
        } else {
#pragma unroll
          for (int h = 0; h < BN / 128; ++h) {
            int mi, row;
            b_source<BN, false>(g, nt, h, mi, row);
            tma_load_2d(sbase + s * C::kStage + C::kABytes + h * 16384u, &maps.b[mi], bar_full(s),
                        kb * BK, row, pol_w);
          }
        }
      };
      const int npre = min(S, it1 - it0);
      {
        SegIter pi{it0, it1, g.kb};
        int unit, k0, k1, n = 0;
        while (n < npre && pi.next(unit, k0, k1)) {
          int mt, nt;
          unit_tile(g, unit, rank, mt, nt);
          for (int kb = k0; kb < k1 && n < npre; ++kb, ++n) {
            // the pair leader expects both CTAs' bytes
            if (prank == 0) mbar_arrive_expect_tx(bar_full(n), PAIR ? 2 * C::kStage : C::kStage);
            load_w(n, nt, kb);
          }
        }
      }
      grid_dep_wait();
      PDS_GEMM_TRACE_HOOK(cta, 1);
      SegIter si{it0, it1, g.kb};
      int unit, k0, k1;
      int mt = 0, nt = 0;
      bool ok = true;
      while (ok && si.next(unit, k0, k1)) {
        unit_tile(g, unit, rank, mt, nt);
        // the last tile's residual, on its way to L2 while the tile is computed
        if (EPI == kEpiResid && si.it >= si.end)
          for (int b = 0; b < C::kResBoxes; ++b)
            tma_prefetch_l2_2d(&maps.e[0], nt * BN + b * 32, mt * BM);
        for (int kb = k0; kb < k1; ++kb) {
          const int s = issued % S;
          if (issued >= npre) {
            if (!mbar_wait(bar_empty(s), ((issued / S) & 1) ^ 1, abort_flag, g.status)) {
              ok = false;
              break;
            }
            if (prank == 0) mbar_arrive_expect_tx(bar_full(s), PAIR ? 2 * C::kStage : C::kStage);
            load_w(s, nt, kb);
          }
          if constexpr (PAIR) {
            tma_load_2d_pair(sbase + s * C::kStage, &maps.a, full_bar(s), kb * BK, mt * BM, pol_a);
          } else {
            tma_load_2d(sbase + s * C::kStage, &maps.a, bar_full(s), kb * BK, mt * BM, pol_a);
          }
          ++issued;
        }
      }
      // The last tile's residual, into the stages as the last MMAs free them
      // (continuing the ring as if they were further k-blocks).  A split
      // tile's residual is loaded too: this CTA may be the one to finish it.
      // (a row-split CTA's epilogue reads the residual rows it finishes itself)
      if (EPI == kEpiResid && ok && it1 > it0 && !RSPLIT) {
        const uint64_t pol_r = policy_evict_first();  // the residual's last read
        // the whole tile's boxes, or the slice this CTA finishes in a split
        int rfirst = 0, rcount = C::kResBoxes;
        if (g.split > 1) {
          const SplitSlice sl = split_slice(g.split, static_cast<int>(crank >> 1));
          rfirst = sl.first;
          rcount = sl.count;
        }
        const int rstages = (rcount + C::kBoxesPerStage - 1) / C::kBoxesPerStage;
        int issued_res = 0;
        for (int f = 0; f < rstages; ++f) {
          const int v = issued + f;
          const int s = v % S;
          if (v >= S && !mbar_wait(bar_empty(s), ((v / S) & 1) ^ 1, abort_flag, g.status)) break;
          const int nb = min(C::kBoxesPerStage, rcount - f * C::kBoxesPerStage);
          mbar_arrive_expect_tx(bar_res0 + 8u * f, static_cast<uint32_t>(nb) * 16384u);
          for (int b = 0; b < nb; ++b)
            tma_load_2d(sbase + s * C::kStage + b * 16384u, &maps.e[0], bar_res0 + 8u * f,
                        nt * BN + (rfirst + f * C::kBoxesPerStage + b) * 32, mt * BM, pol_r);
          ++issued_res;
        }
        // none of these copies may still be landing when the CTA exits,
        // whether or not the epilogue uses them
        for (int f = 0; f < issued_res; ++f)
          if (!mbar_wait(bar_res0 + 8u * f, 0, abort_flag, g.status)) break;
      }
    }
  } else if (warp == 1) {
    setmaxnreg_dec<kRegsControl>();
    if (lane == 0 && prank == 0) {
      SegIter si{it0, it1, g.kb};
      int tile, k0, k1, sg = 0;
      bool ok = true;
      while (ok && si.next(tile, k0, k1)) {
        const int ab = sg & 1;
        if (!mbar_wait(bar_tempty(ab), ((sg >> 1) & 1) ^ 1, abort_flag, g.status)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + ab * BN;
        for (int kb = k0; kb < k1; ++kb) {
          const int s = consumed % S;
          if (!mbar_wait(bar_full(s), (consumed / S) & 1, abort_flag, g.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (consumed == 0) PDS_GEMM_TRACE_HOOK(cta, 2);
          const uint32_t a_addr = sbase + s * C::kStage;
          const uint64_t ad = smem_desc_sw128(a_addr);
          const uint64_t bd = smem_desc_sw128(a_addr + C::kABytes);
#pragma unroll
          for (int k = 0; k < BK / 16; ++k) {
            if constexpr (PAIR) {
              umma_bf16_pair(d_tmem, ad + 2u * k, bd + 2u * k, kIdesc, (kb > k0 || k > 0) ? 1u : 0u);
            } else {
              umma_bf16(d_tmem, ad + 2u * k, bd + 2u * k, kIdesc, (kb > k0 || k > 0) ? 1u : 0u);
            }
          }
          if constexpr (PAIR) {
            umma_commit_pair_mc(bar_empty(s), pmask);  // the stage is free in both CTAs
          } else {
            umma_commit(bar_empty(s));
          }
          ++consumed;
        }
        if (!ok) break;
        if constexpr (PAIR) {
          umma_commit_pair_mc(bar_tfull(ab), pmask);  // both halves of the accumulator
        } else {
          umma_commit(bar_tfull(ab));
        }
        PDS_GEMM_TRACE_HOOK(cta, 3);
        ++sg;
      }
      // Every MMA this thread issued has completed before TMEM is released.
      if constexpr (PAIR) {
        umma_commit_pair(bar_drain);
      } else {
        umma_commit(bar_drain);
      }
      int dummy_abort = 0;
      mbar_wait(bar_drain, 0, &dummy_abort, g.status);
    }
  } else if (warp >= kEpiFirstThread / 32) {
    setmaxnreg_inc<kRegsEpilogue>();
    const int ew = warp - kEpiFirstThread / 32;  // epilogue warp 0..7
    const Stage st{reinterpret_cast<float4*>(smem + S * C::kStage + C::kMiscBytes) + ew * 256};
    const int lane_grp = warp & 3;  // this warp's TMEM lanes: 32*lane_grp ..
    const int ch = ew >> 2;         // which half of the tile's columns
    const int row = lane_grp * 32 + lane;
    const bool leader = threadIdx.x == kEpiFirstThread;
    grid_dep_wait();
    SegIter si{it0, it1, g.kb};
    int unit, k0, k1, sg = 0;
    while (si.next(unit, k0, k1)) {
      const int ab = sg & 1;
      int mt, nt;
      unit_tile(g, unit, rank, mt, nt);
      // the row's RMSNorm scale, read while the accumulator is still being made
      float rscale = 0.f;
      RopeRegs rr;
      if constexpr (EPI == kEpiSwiglu) {
        if (mt * BM + row < g.M) rscale = row_scale(g.swiglu.rs, mt * BM + row);
      } else if constexpr (EPI == kEpiQkv) {
        if (mt * BM + row < g.M) rscale = row_scale(g.qkv.rs, mt * BM + row);
        // (a small tile loads the table after its reduction: see below)
        if (PAIR || (g.M - mt * BM > kSmallRows && !RSPLIT))
          rope_prefetch<BN>(g, nt, ch, mt * BM + row, rr);
      } else if constexpr (EPI == kEpiQkvX) {
        if (mt * BM + row < g.M) rscale = row_scale(g.qkv.rs, mt * BM + row);
      } else if constexpr (EPI == kEpiResid) {
        // the last tile's epilogue goes through shared memory and reads its gains there
        if (si.it >= si.end)
          resid_gain_prefetch<BN>(g, nt, reinterpret_cast<float*>(smem + S * C::kStage + 1024),
                                  static_cast<int>(threadIdx.x) - kEpiFirstThread);
      }
      if (!mbar_wait(bar_tfull(ab), (sg >> 1) & 1, abort_flag, g.status)) break;
      tc_fence_after();
      if (leader) PDS_GEMM_TRACE_HOOK(cta, 4);
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(lane_grp * 32) << 16) + ab * BN;
      const int tile = mt + nt * g.tiles_m;
      Fixup fx{false, 0, 0, grp, rank, unit};
      bool run = true;
      if constexpr (EPI == kEpiResid && PAIR && BN == 256) {
        if (g.split > 1) {
          // the CTA's only tile, finished with the cluster's other pairs
          const bool ok = split_resid_epilogue<BN>(
              g, maps, taddr, mt, nt, row, ch, lane, smem, sbase, grp, bar_res0, bar_ready, bar_recv,
              abort_flag, st, reinterpret_cast<float*>(smem + S * C::kStage + 1024), crank, leader);
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_cluster(mapa_shared(bar_tempty(ab), lead));
          if (!ok) break;
          ++sg;
          continue;
        }
      }
      // rows of the warp's 32 its epilogue stores
      int wlo = 0, whi = 32;
      bool gave_up = false;
      if constexpr (!PAIR) {
        if constexpr (RSPLIT) {
          // the CTA's only tile: exchange rows with the cluster, then the
          // epilogue of the rows this CTA finishes
          const int me = static_cast<int>(crank), R = rsplit_rows(g.rsplit);
          gave_up = !rsplit_exchange<BN, EPI>(g, taddr, row, ch, lane, smem, sbase, bar_ready,
                                              bar_recv, abort_flag, me, leader);
          wlo = max(0, me * R - lane_grp * 32);
          whi = min(32, me * R + R - lane_grp * 32);
          run = !gave_up && wlo < whi;
          if constexpr (EPI == kEpiQkv) {
            if (run) rope_prefetch<BN>(g, nt, ch, mt * BM + row, rr);
          }
        }
      }
      if (!RSPLIT && !(k0 == 0 && k1 == g.kb)) {
        const int slot = (it0 / g.kb == unit) ? 0 : 1;
        float4* mine = reinterpret_cast<float4*>(g.partials) +
                       static_cast<size_t>(cta * 2 + slot) * (BM * BN / 4);
        constexpr int kOwned = owned_chunks<BN, EPI>();
#pragma unroll 1
        for (int i = 0; i < kOwned; ++i) {
          const int j = owned_chunk<BN, EPI>(ch, i);
          if (!chunk_exists<BN, EPI>(g, nt, j)) continue;
          float v[32];
          tmem_load32(taddr + j * 32, v);
          if (mt * BM + row < g.M) {
#pragma unroll
            for (int q = 0; q < 8; ++q)
              __stcg(mine + (j * 8 + q) * BM + row,
                     make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]));
          }
        }
        __threadfence();
        named_bar_sync(1, kEpiThreads);
        if (leader) misc[1] = atomicAdd(&g.counters[tile], 1u);
        named_bar_sync(1, kEpiThreads);
        const int arrived = static_cast<int>(misc[1]);
        const int gf = group_of_iter(g, unit * g.kb), gl = group_of_iter(g, unit * g.kb + g.kb - 1);
        if (arrived == gl - gf) {
          __threadfence();
          fx = Fixup{true, gf, gl, grp, rank, unit};
        } else {
          run = false;
        }
      }
      if (run) {
        const bool last = si.it >= si.end;
        const bool split = fx.active;
        // A split tile is first finished in TMEM (the other contributors'
        // partials added in k order), then the epilogue reads TMEM as for an
        // unsplit tile.  The CTA's last tile stages the partials in the
        // drained stages (after the residual boxes of a residual GEMM).
        // (a pair tile has two full row tiles: never a small one)
        if (!PAIR && split && g.M - mt * BM <= kSmallRows) {
          if constexpr (!PAIR)
            fixup_reduce_small<BN, EPI>(g, fx, taddr, mt, nt, row, ch,
                                        static_cast<int>(threadIdx.x) - kEpiFirstThread,
                                        reinterpret_cast<float4*>(smem + S * C::kStage + C::kMiscBytes));
        } else if (split) {
          const bool row_ok = mt * BM + row < g.M;
          if (last) {
            fixup_reduce_smem<BN, EPI, PAIR>(g, fx, taddr, nt, row, ch, smem, sbase, it1 - it0,
                                             EPI == kEpiResid ? C::kResBoxes : 0, row_ok);
          } else {
            fixup_reduce_regs<BN, EPI>(g, fx, taddr, nt, row, ch, row_ok);
          }
          fx.active = false;
        }
        if constexpr (EPI == kEpiQkv && !PAIR) {
          if (g.M - mt * BM <= kSmallRows) rope_prefetch<BN>(g, nt, ch, mt * BM + row, rr);
        }
        if (EPI == kEpiResid && last && !RSPLIT) {
          auto acc = [&](int j, float (&v)[32]) { tmem_load32(taddr + j * 32, v); };
          if (!resid_epilogue_smem<BN, PAIR>(g, maps, mt, nt, row, ch, lane, smem, sbase, it1 - it0,
                                             bar_res0, abort_flag, st,
                                             reinterpret_cast<float*>(smem + S * C::kStage + 1024),
                                             ch * (BN / 64), BN / 64, 0, acc))
            break;
        } else {
          run_epilogue<BN, EPI>(g, taddr, mt, nt, row, ch, lane, rscale, st, rr, wlo, whi);
        }
        if (split && leader) g.counters[tile] = 0;
      }
      if (leader) PDS_GEMM_TRACE_HOOK(cta, 5);
      // this warp's TMEM reads are done: one arrival per warp, on the pair
      // leader's barrier for a pair
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (PAIR && prank != 0) {
          mbar_arrive_cluster(mapa_shared(bar_tempty(ab), lead));
        } else {
          mbar_arrive(bar_tempty(ab));
        }
      }
      if (gave_up) break;
      ++sg;
    }
  } else {
    setmaxnreg_dec<kRegsControl>();  // warps 2 and 3: only their registers are needed
  }

  // On a timeout the producer may have loads in flight: give them time to
  // land (they complete in microseconds) before the shared memory is released.
  if (warp == 0 && lane == 0 && *abort_flag) {
    const uint64_t t0 = global_timer_ns();
    while (global_timer_ns() - t0 < 200000ull) {
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // no CTA leaves while a peer may still copy into it or arrive on it
  if (g.cs > 1) cluster_sync();
  if (threadIdx.x == 0) PDS_GEMM_TRACE_HOOK(cta, 6);
  if (warp == 1) {
    if constexpr (PAIR) {
      tmem_dealloc_pair(tmem_base, C::kTmemCols);
    } else {
      tmem_dealloc(tmem_base, C::kTmemCols);
    }
  }
}

// ------------------------------------------------------------ host side

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return static_cast<EncodeTiledFn>(nullptr);
    return reinterpret_cast<EncodeTiledFn>(p);
  }();
  return fn;
}

}  // namespace

struct TmapKey {
  const void* p;
  uint64_t inner, outer;
  uint32_t box_inner, box_rows, elem_bytes;
  bool operator==(const TmapKey& o) const {
    return p == o.p && inner == o.inner && outer == o.outer && box_inner == o.box_inner &&
           box_rows == o.box_rows && elem_bytes == o.elem_bytes;
  }
};
struct TmapKeyHash {
  size_t operator()(const TmapKey& k) const {
    return std::hash<const void*>()(k.p) ^ (k.inner * 0x9E3779B97F4A7C15ull) ^ (k.outer << 20) ^
           (static_cast<size_t>(k.box_rows) << 44) ^ (static_cast<size_t>(k.box_inner) << 32) ^
           (static_cast<size_t>(k.elem_bytes) << 56);
  }
};
struct TmapCache {
  std::mutex mu;
  std::unordered_map<TmapKey, CUtensorMap, TmapKeyHash> maps;
};

TmapCache* tmap_cache_create() { return new TmapCache(); }
void tmap_cache_destroy(TmapCache* c) { delete c; }

namespace {

// Row-major matrix [outer rows, inner columns] of bf16 (elem_bytes 2) or
// float32 (4), box of box_inner columns (128 bytes) x box_rows rows, 128-byte
// swizzle.  The default is the GEMM operand box: 64 bf16 columns x 128 rows.
pds_status get_map(TcContext& c, CUtensorMap* out, const void* p, uint64_t inner, uint64_t outer,
                   std::string* err, uint32_t box_rows = 128, uint32_t elem_bytes = 2) {
  const uint32_t box_inner = 128u / elem_bytes;
  TmapKey key{p, inner, outer, box_inner, box_rows, elem_bytes};
  if (c.maps) {
    std::lock_guard<std::mutex> g(c.maps->mu);
    auto it = c.maps->maps.find(key);
    if (it != c.maps->maps.end()) {
      *out = it->second;
      return PDS_OK;
    }
  }
  EncodeTiledFn fn = encode_fn();
  if (!fn) {
    *err = "cuTensorMapEncodeTiled is not available from the driver";
    return PDS_ELAUNCH;
  }
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {inner * elem_bytes};
  const cuuint32_t box[2] = {box_inner, box_rows};
  const cuuint32_t es[2] = {1, 1};
  const CUtensorMapDataType dt =
      elem_bytes == 4 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  CUresult r = fn(out, dt, 2, const_cast<void*>(p), dims, strides, box,
                  es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    *err = "cuTensorMapEncodeTiled failed (" + std::to_string(static_cast<int>(r)) + ")";
    return PDS_ELAUNCH;
  }
  if (c.maps) {
    std::lock_guard<std::mutex> g(c.maps->mu);
    c.maps->maps.emplace(key, *out);
  }
  return PDS_OK;
}

// Shared memory a row-split CTA of a cluster of c needs in its drained
// stages (the worst CTA of the cluster): the other CTAs' slices of its rows
// and a box per 32-column chunk of each lane group it sends rows from.
int rsplit_stage_bytes(int bn, int c) {
  const int R = rsplit_rows(c);
  int worst = 0;
  for (int me = 0; me < c; ++me) {
    const int lo = me * R, hs = std::min(BM, lo + R);
    int slots = 0;
    for (int l = 0; l < BM / 32; ++l) slots += (32 * l < lo || 32 * l + 32 > hs) ? 1 : 0;
    worst = std::max(worst, (c - 1) * R * bn * 4 + slots * bn * 128);
  }
  return worst;
}

void make_schedule(GemmArgs& g, const TcContext& c, int M, int tiles_n, int K, int bn,
                   int max_grid = kGemmMaxGrid, bool allow_pair = true, int split = 0,
                   bool allow_rsplit = true) {
  g.M = M;
  g.K = K;
  g.tiles_m = (M + BM - 1) / BM;
  g.tiles_n = tiles_n;
  g.kb = K / BK;
  // Group size: all row tiles of a column tile (up to 8), a divisor of tiles_m.
  int gs = std::min(g.tiles_m, 8);
  while (g.tiles_m % gs) --gs;
  g.gs = gs;
  g.mgs = g.tiles_m / gs;
  g.units = g.mgs * g.tiles_n;
  g.total = g.units * g.kb;
  // Pair mode for 256-wide tiles whenever the group holds whole pairs of
  // row tiles: it halves the weight bytes each SM takes in per k-block.
  // Otherwise every CTA runs alone (clusters of one).
  g.cs = 1;
  g.pair = 0;
  g.split = 0;
  g.rsplit = 0;
  if (bn == 256 && gs % 2 == 0 && allow_pair && split != 0) {
    // Cluster split-K (residual epilogues only; split = 0 elsewhere): one
    // cluster of 2S CTAs per 256-row pair tile when the pair tiles alone
    // would leave at least half of the SMs idle.  split < 0 picks the
    // largest S (at most 4) whose CTAs fit one per SM; split > 0 caps it.
    const int ctas = std::min({c.num_sms > 0 ? c.num_sms : 148, kGemmMaxGrid, max_grid});
    const int units = (g.tiles_m / 2) * tiles_n;
    int S = 1;
    for (int t = 4; t >= 2; --t)
      if (2 * t * units <= ctas && t <= g.kb && (split < 0 || t <= split)) {
        S = t;
        break;
      }
    if (S >= 2) {
      g.gs = 2;
      g.mgs = g.tiles_m / 2;
      g.units = units;
      g.total = units * g.kb;
      g.groups = S * units;
      g.grid = 2 * g.groups;
      g.pair = 1;
      g.cs = 2 * S;
      g.split = S;
      return;
    }
  }
  if (bn == 256 && gs % 2 == 0 && allow_pair) {
    g.pair = 1;
    g.cs = 2;
  }
  const int ctas = std::min({c.num_sms > 0 ? c.num_sms : 148, kGemmMaxGrid, max_grid});
  const int gmax = std::max(1, std::min(ctas / gs, g.total / kMinItersPerCta));
  if (g.tiles_m == 1 && M <= kSmallRows) {
    // A decode batch: the split tiles' partials are a few rows, reduced by
    // all epilogue threads at once (fixup_reduce_small), so every column tile
    // gets as many CTAs as fill the GPU, each an equal k range -- an aligned
    // one (c dividing the k-blocks, every CTA on one tile) unless that costs
    // more than a quarter of the CTAs.
    const int c_max = std::max(1, std::min(ctas / g.tiles_n, g.kb / kMinItersPerCta));
    int c = c_max;
    for (int d = c_max; d >= 1; --d)
      if (g.kb % d == 0) {
        if (4 * d >= 3 * c_max) c = d;
        break;
      }
    g.groups = g.tiles_n * c;
    g.grid = g.groups * gs;
    return;
  }
  if (g.tiles_m == 1 && allow_rsplit) {
    // A single row tile of more rows streams every weight byte once and is
    // bound by how fast its CTAs pull weights in (a CTA keeps its stages'
    // bytes in flight, no more): it wants many CTAs on each tile, which the
    // row-split cluster gives without a serial reduction -- each of the c
    // CTAs of a tile's cluster takes 1/c of the k-blocks and finishes 1/c
    // of the rows.  The largest c in 3..8 that leaves every CTA two
    // k-blocks, keeps all clusters on the GPU at once and whose exchange
    // fits the drained stages (c <= 4 for 256-wide tiles).  (Measured at
    // M = 128 on GB300: a split in two lost to the unsplit schedule, whose
    // CTAs are then one per column tile.)
    const int stage_bytes = bn == 256 ? Cfg<256>::kStages * static_cast<int>(Cfg<256>::kStage)
                                      : Cfg<128>::kStages * static_cast<int>(Cfg<128>::kStage);
    for (int cc = 8; cc >= 3; --cc) {
      if (2 * cc > g.kb || g.tiles_n * cc > ctas || rsplit_stage_bytes(bn, cc) > stage_bytes)
        continue;
      g.rsplit = cc;
      g.cs = cc;
      g.groups = g.tiles_n * cc;
      g.grid = g.groups;
      return;
    }
  }
  if (g.tiles_m == 1) {
    // A single row tile streams every weight byte once and is bound by how
    // fast the CTAs pull weights in, which wants many CTAs; but each extra
    // CTA on a tile adds a partial tile to the finisher's serial reduction.
    // Measured on GB300 at M = 128 (Llama-3.2-1B shapes): splits that give
    // every tile the same number c of CTAs, c dividing the k-blocks, with
    // about 64 CTAs in all, beat using every SM by 1.3-2.2x per GEMM.
    int best_c = 0;
    for (int cc = 1; g.tiles_n * cc <= ctas && cc * kMinItersPerCta <= g.kb; cc *= 2) {
      if (g.kb % cc) continue;
      if (!best_c || std::abs(g.tiles_n * cc - kSingleRowCtas) <
                         std::abs(g.tiles_n * best_c - kSingleRowCtas))
        best_c = cc;
    }
    g.groups = best_c ? g.tiles_n * best_c : gmax;
    g.grid = g.groups * gs;
    return;
  }
  // Pick the group count by a cost model measured on GB300 for these tiles:
  // about 0.35 us per k-block of a group's range, plus, when units are split
  // across groups, about 4 us + 5 us per extra contributor for storing,
  // reducing and re-reading partial tiles.  Fewer CTAs without splits often win.
  // A 128-wide tile moves two thirds of the shared-memory bytes of a 256-wide
  // one per k-block, and its k-blocks take about that much less time.
  const double kb_us = bn == 256 ? 0.35 : 0.24;
  constexpr double kSplitUs = 4.0, kSplitPerContribUs = 5.0;
  double best = 1e30;
  int best_g = gmax;
  for (int gr = gmax; gr >= std::max(1, gmax / 3); --gr) {
    const double per = static_cast<double>(g.total) / gr;
    double cost = std::ceil(per) * kb_us;
    if (g.units % gr != 0) {
      const bool aligned = g.total % gr == 0 && (g.kb % static_cast<int>(per) == 0);
      const double contrib = g.kb / per + (aligned ? 0.0 : 1.0);
      cost += kSplitUs + kSplitPerContribUs * std::max(0.0, contrib - 1.0);
    }
    if (cost < best - 1e-9) {
      best = cost;
      best_g = gr;
    }
  }
  g.groups = best_g;
  g.grid = g.groups * gs;
}

template <int BN, int EPI, bool PAIR, bool RSPLIT>
pds_status launch_impl(TcContext& c, const GemmMaps& maps, GemmArgs& g, cudaStream_t st,
                       std::string* err) {
  using Cf = Cfg<BN, PAIR>;
  const void* fn = reinterpret_cast<const void*>(gemm_kernel<BN, EPI, PAIR, RSPLIT>);
  const cudaError_t attr_err = kernel_smem_attr(fn, static_cast<int>(Cf::kSmem));
  if (attr_err != cudaSuccess) {
    *err = std::string("gemm shared-memory attribute: ") + cudaGetErrorString(attr_err);
    return PDS_ELAUNCH;
  }
  const size_t part_bytes = static_cast<size_t>(kGemmMaxGrid) * 2 * BM * 256 * sizeof(float);
  if (c.ws_bytes < part_bytes + static_cast<size_t>(g.tiles_m) * g.tiles_n * 4) {
    *err = "GEMM scratch too small";
    return PDS_EINVAL;
  }
  g.status = c.status;
  g.partials = reinterpret_cast<float*>(c.ws);
  g.counters = reinterpret_cast<uint32_t*>(c.ws + part_bytes);

  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = Cf::kSmem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  int na = 0;
  if (g.cs > 1) {
    // never more clusters than fit on the GPU at once (one CTA per SM)
    auto fit = [&](int cs) { return std::max(1, kernel_max_clusters(fn, cfg, cs)); };
    if (g.split > 1) {
      // all of a split GEMM's clusters at once, or fewer pairs per tile
      int S = g.split;
      while (S >= 2 && fit(2 * S) < g.units) --S;
      if (S != g.split) {
        if (S >= 2) {
          g.split = S;
          g.cs = 2 * S;
          g.groups = S * g.units;
          g.grid = 2 * g.groups;
        } else {
          make_schedule(g, c, g.M, g.tiles_n, g.K, BN, kGemmMaxGrid, true, 0);
        }
      }
    }
    if constexpr (RSPLIT) {
      // every tile's cluster at once, or fewer CTAs per tile
      int cc = g.rsplit;
      while (cc >= 3 && fit(cc) < g.tiles_n) --cc;
      if (cc != g.rsplit) {
        if (cc >= 3) {
          g.rsplit = cc;
          g.cs = cc;
          g.groups = g.tiles_n * cc;
          g.grid = g.groups;
        } else {
          make_schedule(g, c, g.M, g.tiles_n, g.K, BN, kGemmMaxGrid, false, 0, false);
          return launch_impl<BN, EPI, false, false>(c, maps, g, st, err);
        }
      }
    }
    if (g.cs > 1 && g.split < 2 && g.rsplit < 2) {
      const int cap_groups = std::max(1, fit(g.cs) * g.cs / g.gs);
      if (g.groups > cap_groups) {
        g.groups = cap_groups;
        g.grid = g.groups * g.gs;
      }
    }
    if (g.cs > 1) {
      attr[na].id = cudaLaunchAttributeClusterDimension;
      attr[na].val.clusterDim.x = g.cs;
      attr[na].val.clusterDim.y = 1;
      attr[na].val.clusterDim.z = 1;
      ++na;
    }
  }
  if (c.pdl) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  cfg.gridDim = dim3(g.grid);
  cfg.attrs = attr;
  cfg.numAttrs = na;
  cudaError_t ce = cudaLaunchKernelEx(&cfg, gemm_kernel<BN, EPI, PAIR, RSPLIT>, maps, g);
  if (ce != cudaSuccess) {
    *err = std::string("gemm launch: ") + cudaGetErrorString(ce);
    return PDS_ELAUNCH;
  }
  return PDS_OK;
}

template <int BN, int EPI>
pds_status launch(TcContext& c, const GemmMaps& maps, GemmArgs& g, cudaStream_t st,
                  std::string* err) {
  if constexpr (BN == 256) {
    if (g.pair) return launch_impl<BN, EPI, true, false>(c, maps, g, st, err);
  }
  if (g.rsplit > 1) return launch_impl<BN, EPI, false, true>(c, maps, g, st, err);
  return launch_impl<BN, EPI, false, false>(c, maps, g, st, err);
}

}  // namespace

cudaError_t kernel_smem_attr(const void* fn, int bytes) {
  static std::mutex mu;
  static std::map<std::pair<const void*, int>, cudaError_t> done;
  int dev = 0;
  cudaError_t ce = cudaGetDevice(&dev);
  if (ce != cudaSuccess) return ce;
  std::lock_guard<std::mutex> lock(mu);
  auto it = done.find({fn, dev});
  if (it != done.end()) return it->second;
  ce = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  done[{fn, dev}] = ce;
  return ce;
}

int kernel_max_clusters(const void* fn, const cudaLaunchConfig_t& cfg, int cs) {
  static std::mutex mu;
  static std::map<std::tuple<const void*, int, int>, int> done;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  std::lock_guard<std::mutex> lock(mu);
  auto it = done.find({fn, dev, cs});
  if (it != done.end()) return it->second;
  cudaLaunchAttribute ca[1];
  ca[0].id = cudaLaunchAttributeClusterDimension;
  ca[0].val.clusterDim.x = cs;
  ca[0].val.clusterDim.y = 1;
  ca[0].val.clusterDim.z = 1;
  cudaLaunchConfig_t q = cfg;
  q.gridDim = dim3(cs);
  q.attrs = ca;
  q.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, fn, &q) != cudaSuccess || n < 0) {
    cudaGetLastError();
    n = 0;
  }
  done[{fn, dev, cs}] = n;
  return n;
}

pds_status tc_map_bf16(TcContext& c, CUtensorMap* out, const void* p, uint64_t inner,
                       uint64_t outer, uint32_t box_rows, std::string* err) {
  return get_map(c, out, p, inner, outer, err, box_rows, 2);
}

size_t tc_gemm_scratch_bytes(int M, int max_tiles_n) {
  const size_t part_bytes = static_cast<size_t>(kGemmMaxGrid) * 2 * BM * 256 * sizeof(float);
  const size_t tiles = static_cast<size_t>((M + BM - 1) / BM) * max_tiles_n;
  return part_bytes + ((tiles * 4 + 255) / 256) * 256;
}

pds_status tc_gemm_plain(TcContext& c, const uint16_t* A, const uint16_t* W, float* Cout, int M,
                         int N, int K, cudaStream_t st, std::string* err) {
  const int bn = N % 256 == 0 ? 256 : 128;
  GemmArgs g{};
  g.wrows0 = N;
  g.wrows1 = 0;
  g.c_out = Cout;
  g.ldc = N;
  make_schedule(g, c, M, N / bn, K, bn);
  GemmMaps maps{};
  pds_status rc;
  if ((rc = get_map(c, &maps.a, A, K, M, err)) != PDS_OK) return rc;
  if ((rc = get_map(c, &maps.b[0], W, K, N, err)) != PDS_OK) return rc;
  maps.b[1] = maps.b[0];
  maps.b[2] = maps.b[0];
  return bn == 256 ? launch<256, kEpiPlain>(c, maps, g, st, err)
                   : launch<128, kEpiPlain>(c, maps, g, st, err);
}

pds_status tc_gemm_resid(TcContext& c, const uint16_t* A, const uint16_t* W, int M, int N, int K,
                         const ResidEpilogue& e, cudaStream_t st, std::string* err) {
  // A single row tile: 128-wide tiles (twice the tiles to spread the
  // weights over; measured faster for both residual GEMMs at M = 128).
  // Pairs of row tiles: 256 x 256 pair tiles (256 x 128 pair tiles without
  // a k split were measured slower at M = 512: a 256 x 128 x 64 pair step
  // took as long as a 256 x 256 x 64 one).
  const int bn = (N % 256 == 0 && M > BM) ? 256 : 128;
  GemmArgs g{};
  g.wrows0 = N;
  g.resid = e;
  g.resid_n = N;
  make_schedule(g, c, M, N / bn, K, bn, kGemmMaxGrid, true, -1);
  GemmMaps maps{};
  pds_status rc;
  if ((rc = get_map(c, &maps.a, A, K, M, err)) != PDS_OK) return rc;
  if ((rc = get_map(c, &maps.b[0], W, K, N, err)) != PDS_OK) return rc;
  maps.b[1] = maps.b[0];
  maps.b[2] = maps.b[0];
  // residual in (whole-tile-high boxes), h and a out (one warp's 32 rows)
  if ((rc = get_map(c, &maps.e[0], e.resid, N, M, err, 128, 4)) != PDS_OK) return rc;
  if ((rc = get_map(c, &maps.e[1], e.out, N, M, err, 32, 4)) != PDS_OK) return rc;
  if (e.gain) {
    if ((rc = get_map(c, &maps.e[2], e.a_out, N, M, err, 32, 2)) != PDS_OK) return rc;
  } else {
    maps.e[2] = maps.e[1];
  }
  return bn == 256 ? launch<256, kEpiResid>(c, maps, g, st, err)
                   : launch<128, kEpiResid>(c, maps, g, st, err);
}

pds_status tc_gemm_swiglu(TcContext& c, const uint16_t* A, const WeightRows& W, int M, int K,
                          const SwigluEpilogue& e, cudaStream_t st, std::string* err) {
  GemmArgs g{};
  g.pair_mode = 1;
  g.swiglu = e;
  make_schedule(g, c, M, e.ffn / 128, K, 256);
  GemmMaps maps{};
  pds_status rc;
  if ((rc = get_map(c, &maps.a, A, K, M, err)) != PDS_OK) return rc;
  if ((rc = get_map(c, &maps.b[0], W.w[0], K, W.rows[0], err)) != PDS_OK) return rc;
  if ((rc = get_map(c, &maps.b[1], W.w[1], K, W.rows[1], err)) != PDS_OK) return rc;
  maps.b[2] = maps.b[0];
  return launch<256, kEpiSwiglu>(c, maps, g, st, err);
}

pds_status tc_gemm_qkv(TcContext& c, const uint16_t* A, const WeightRows& W, int M, int K,
                       const QkvEpilogue& e, cudaStream_t st, std::string* err) {
  GemmArgs g{};
  g.wrows0 = W.rows[0];
  g.wrows1 = W.rows[1];
  g.qkv = e;
  const int N = W.rows[0] + W.rows[1] + W.rows[2];
  // 256-column tiles always (each 128-column half holds whole heads); a
  // last half past N reads zero rows and is skipped by the epilogue.
  make_schedule(g, c, M, (N + 255) / 256, K, 256);
  GemmMaps maps{};
  pds_status rc;
  if ((rc = get_map(c, &maps.a, A, K, M, err)) != PDS_OK) return rc;
  for (int i = 0; i < 3; ++i)
    if ((rc = get_map(c, &maps.b[i], W.w[i], K, W.rows[i], err)) != PDS_OK) return rc;
  const bool general = e.rope_layout != PDS_ROPE_NEOX || e.rot_dim != e.head_dim || e.bias[0] ||
                       e.bias[1] || e.bias[2] || e.norm[0] || e.norm[1];
  return general ? launch<256, kEpiQkvX>(c, maps, g, st, err)
                 : launch<256, kEpiQkv>(c, maps, g, st, err);
}

// ------------------------------------------------ no-allocation GEMM entry
//
// Scratch of tc_gemm_plain_noalloc (the C entry pds_gemm_bf16_noalloc): a
// status word, the stream-K tile counters and the partial tiles, all in
// one array of this module's global memory, so that the call allocates
// nothing.  Every GPU that loads the library holds the array until the
// process exits.  Every call shares it: calls that overlap on one GPU (on
// any streams) race.
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(24) << 20;  // 24 MiB in all
constexpr size_t kNoAllocStatusBytes = 256;
constexpr size_t kNoAllocCounterBytes = size_t(64) << 10;  // 16384 tile counters
constexpr int kNoAllocBN = 128;                            // tiles of 128 x 128
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kNoAllocMaxDevices = 64;
std::mutex g_noalloc_mu;
char* g_noalloc_addr[kNoAllocMaxDevices] = {};

// Device address of the array on the current device.  The name of the
// array in host code is a host-side stand-in, not a device address: the
// address is looked up once per device, with that device current.
pds_status noalloc_scratch(char** out, std::string* err) {
  int dev = 0;
  cudaError_t ce = cudaGetDevice(&dev);
  if (ce != cudaSuccess) {
    *err = std::string("no CUDA device: ") + cudaGetErrorString(ce);
    return PDS_ELAUNCH;
  }
  if (dev < 0 || dev >= kNoAllocMaxDevices) {
    *err = "device ordinal beyond the static-scratch table";
    return PDS_EINVAL;
  }
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_addr[dev]) {
    void* p = nullptr;
    ce = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (ce != cudaSuccess || !p) {
      *err = std::string("static scratch address: ") + cudaGetErrorString(ce);
      return PDS_ELAUNCH;
    }
    g_noalloc_addr[dev] = static_cast<char*>(p);
  }
  *out = g_noalloc_addr[dev];
  return PDS_OK;
}

}  // namespace

size_t tc_gemm_noalloc_max_tiles() { return kNoAllocCounterBytes / 4; }

pds_status tc_noalloc_take_status(uint32_t* flags, std::string* err) {
  *flags = 0;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kNoAllocMaxDevices) return PDS_OK;
  char* base = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    base = g_noalloc_addr[dev];
  }
  if (!base) return PDS_OK;  // no call on this device yet
  cudaError_t ce = cudaMemcpy(flags, base, sizeof(uint32_t), cudaMemcpyDeviceToHost);
  if (ce == cudaSuccess && *flags) ce = cudaMemset(base, 0, sizeof(uint32_t));
  if (ce != cudaSuccess) {
    *err = std::string("static scratch status word: ") + cudaGetErrorString(ce);
    return PDS_ELAUNCH;
  }
  return PDS_OK;
}

pds_status tc_gemm_plain_noalloc(const uint16_t* A, const uint16_t* W, float* Cout, int M, int N,
                                 int K, int num_sms, cudaStream_t st, std::string* err) {
  const size_t tiles = static_cast<size_t>((M + BM - 1) / BM) * (N / kNoAllocBN);
  if (tiles > tc_gemm_noalloc_max_tiles()) {
    *err = "pds_gemm_bf16_noalloc: ceil(M/128) * N/128 = " + std::to_string(tiles) +
           " output tiles exceed the static scratch's " +
           std::to_string(tc_gemm_noalloc_max_tiles());
    return PDS_EINVAL;
  }
  char* base = nullptr;
  pds_status rc = noalloc_scratch(&base, err);
  if (rc != PDS_OK) return rc;
  uint32_t* status = reinterpret_cast<uint32_t*>(base);
  uint32_t* counters = reinterpret_cast<uint32_t*>(base + kNoAllocStatusBytes);
  float* partials = reinterpret_cast<float*>(base + kNoAllocStatusBytes + kNoAllocCounterBytes);
  const size_t per_cta = 2 * static_cast<size_t>(BM) * kNoAllocBN * sizeof(float);
  const int grid_cap = static_cast<int>(
      (kNoAllocScratchBytes - kNoAllocStatusBytes - kNoAllocCounterBytes) / per_cta);

  // The counters are shared with earlier calls: they must start at zero.
  // The status word keeps what earlier calls set until pds_component_sync
  // reads and clears it.
  cudaError_t ce = cudaMemsetAsync(counters, 0, tiles * 4, st);
  if (ce != cudaSuccess) {
    *err = std::string("static scratch counter reset: ") + cudaGetErrorString(ce);
    return PDS_ELAUNCH;
  }
  TcContext c{};
  c.num_sms = num_sms;
  GemmArgs g{};
  g.wrows0 = N;
  g.c_out = Cout;
  g.ldc = N;
  make_schedule(g, c, M, N / kNoAllocBN, K, kNoAllocBN, grid_cap, false, 0, false);
  g.cs = 1;  // a plain launch, without clusters
  GemmMaps maps{};
  if ((rc = get_map(c, &maps.a, A, K, M, err)) != PDS_OK) return rc;
  if ((rc = get_map(c, &maps.b[0], W, K, N, err)) != PDS_OK) return rc;
  maps.b[1] = maps.b[0];
  maps.b[2] = maps.b[0];
  g.status = status;
  g.partials = partials;
  g.counters = counters;

  using Cf = Cfg<kNoAllocBN, false>;
  const cudaError_t attr_err =
      kernel_smem_attr(reinterpret_cast<const void*>(gemm_kernel<kNoAllocBN, kEpiPlain, false, false>),
                       static_cast<int>(Cf::kSmem));
  if (attr_err != cudaSuccess) {
    *err = std::string("gemm shared-memory attribute: ") + cudaGetErrorString(attr_err);
    return PDS_ELAUNCH;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(g.grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = Cf::kSmem;
  cfg.stream = st;
  ce = cudaLaunchKernelEx(&cfg, gemm_kernel<kNoAllocBN, kEpiPlain, false, false>, maps, g);
  if (ce != cudaSuccess) {
    *err = std::string("gemm launch: ") + cudaGetErrorString(ce);
    return PDS_ELAUNCH;
  }
  return PDS_OK;
}

}  // namespace pds
