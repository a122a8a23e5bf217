// Persistent stream-K tcgen05 GEMM with the stack's fused epilogues.
//
//   C[M, N] = A[M, K] . W[N, K]^T      A, W bf16 (K contiguous), fp32 accumulate
//
// One CTA per SM (192 threads, ~193 KB of shared memory, 2*BN TMEM columns):
//   warp 0      TMA producer: A box [128 x 64] and W boxes [128 x 64] per
//               k-block into a ring of S shared-memory stages (128-byte swizzle)
//   warp 1      tcgen05.mma issuer (one thread): 128 x BN x 16 steps into a
//               double-buffered TMEM accumulator; commits free the stages
//   warps 2..5  epilogue: tcgen05.ld of the accumulator (one TMEM lane = one
//               output row per thread), fused epilogue, global stores
//
// Work split (stream-K): the tiles x k-blocks iteration space is cut into
// `grid` equal contiguous ranges, one per CTA.  A tile whose k-blocks are
// spread over several CTAs is finished by the last of them to arrive: each
// stores its float32 partial tile to scratch and bumps the tile's counter;
// the one that sees the final count adds all partials in CTA order (hence
// in k order: the sum is the same whoever arrives last) and runs the
// epilogue.  No CTA ever waits for another.
//
// Epilogues (the stack's fusions; frink-models 0.29.0
// src/decoder/cuda_prefill.rs, module doc: everything between the seven
// matmuls of a layer is a kernel):
//   plain   store float32 C
//   resid   h = resid + acc; store h; a = bf16(h * gain); per-128-column
//           sum of squares of h (the next RMSNorm's statistics)
//   swiglu  act = silu(r*g) * (r*u): W rows of a tile are 128 gate rows then
//           the same 128 up rows; r = rsqrt(mean sum-of-squares + eps)
//   qkv     r-scaled q|k|v; NeoX RoPE of q and k from a (cos, sin) table;
//           q to the workspace, k and v rows into the caches at start_pos+b
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstring>
#include <mutex>
#include <unordered_map>

#include "sm100.cuh"
#include "tc.h"

namespace pds {

namespace {

enum EpiKind { kEpiPlain = 0, kEpiResid = 1, kEpiSwiglu = 2, kEpiQkv = 3 };

constexpr int BM = 128;
constexpr int BK = 64;
constexpr int kMinItersPerCta = 4;

struct GemmMaps {
  CUtensorMap a;
  CUtensorMap b[3];
};

struct GemmArgs {
  int M, K;
  int tiles_m, tiles_n, kb, total, grid;
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

template <int BN>
struct Cfg {
  static constexpr int kStages = BN == 256 ? 4 : 6;
  static constexpr uint32_t kABytes = BM * BK * 2;
  static constexpr uint32_t kBBytes = BN * BK * 2;
  static constexpr uint32_t kStage = kABytes + kBBytes;
  static constexpr uint32_t kTmemCols = 2 * BN;
  static constexpr int kBars = 2 * kStages + 5;
  static constexpr size_t kSmem = 1024 + kStages * kStage + kBars * 8 + 16;
};

__device__ __forceinline__ int seg_begin(const GemmArgs& g, int c) {
  return static_cast<int>((static_cast<long long>(c) * g.total) / g.grid);
}
// The CTA whose range holds iteration i.
__device__ __forceinline__ int cta_of_iter(const GemmArgs& g, int i) {
  return static_cast<int>(((static_cast<long long>(i) + 1) * g.grid - 1) / g.total);
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

template <int BN>
__device__ __forceinline__ void b_source(const GemmArgs& g, int nt, int h, int& mi, int& row) {
  if (g.pair_mode) {
    mi = h;
    row = nt * 128;
    return;
  }
  const int n0 = nt * BN + h * 128;
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

struct Fixup {
  bool active;
  int cf, cl, me, tile;
};

// Chunk j (32 columns) of this thread's accumulator row, plus the partial
// tiles of the other CTAs of a split tile, summed in CTA order.
template <int BN>
__device__ __forceinline__ void load_chunk(const GemmArgs& g, uint32_t taddr, const Fixup& fx,
                                           int j, int row, float (&v)[32]) {
  sm100::tmem_load32(taddr + j * 32, v);
  if (!fx.active) return;
  float own[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    own[i] = v[i];
    v[i] = 0.f;
  }
  for (int c = fx.cf; c <= fx.cl; ++c) {
    if (c == fx.me) {
#pragma unroll
      for (int i = 0; i < 32; ++i) v[i] += own[i];
    } else {
      const int slot = (seg_begin(g, c) / g.kb == fx.tile) ? 0 : 1;
      const float4* p = reinterpret_cast<const float4*>(g.partials) +
                        static_cast<size_t>(c * 2 + slot) * (BM * BN / 4);
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const float4 x = __ldcg(p + (j * 8 + q) * BM + row);
        v[4 * q] += x.x;
        v[4 * q + 1] += x.y;
        v[4 * q + 2] += x.z;
        v[4 * q + 3] += x.w;
      }
    }
  }
}

__device__ __forceinline__ void store_bf16x32(uint16_t* dst, const float (&v)[32]) {
  uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    d4[q] = make_uint4(pack_bf16x2(v[8 * q], v[8 * q + 1]), pack_bf16x2(v[8 * q + 2], v[8 * q + 3]),
                       pack_bf16x2(v[8 * q + 4], v[8 * q + 5]),
                       pack_bf16x2(v[8 * q + 6], v[8 * q + 7]));
  }
}

template <int BN, int EPI>
__device__ __forceinline__ void run_epilogue(const GemmArgs& g, uint32_t taddr, const Fixup& fx,
                                             int m, int nt, int row) {
  const bool live = m < g.M;
  if constexpr (EPI == kEpiPlain) {
    for (int j = 0; j < BN / 32; ++j) {
      float v[32];
      load_chunk<BN>(g, taddr, fx, j, row, v);
      if (live) {
        float4* d4 = reinterpret_cast<float4*>(g.c_out + static_cast<size_t>(m) * g.ldc + nt * BN +
                                               j * 32);
#pragma unroll
        for (int q = 0; q < 8; ++q)
          d4[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
      }
    }
  } else if constexpr (EPI == kEpiResid) {
    const ResidEpilogue& e = g.resid;
    const int N = g.resid_n;
    for (int gq = 0; gq < BN / 128; ++gq) {
      float ss = 0.f;
      for (int jj = 0; jj < 4; ++jj) {
        const int j = gq * 4 + jj;
        const int n = nt * BN + j * 32;
        float v[32];
        load_chunk<BN>(g, taddr, fx, j, row, v);
        if (live) {
          const size_t off = static_cast<size_t>(m) * N + n;
          const float4* r4 = reinterpret_cast<const float4*>(e.resid + off);
          float4* o4 = reinterpret_cast<float4*>(e.out + off);
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            float4 x = r4[q];
            x.x += v[4 * q];
            x.y += v[4 * q + 1];
            x.z += v[4 * q + 2];
            x.w += v[4 * q + 3];
            o4[q] = x;
            v[4 * q] = x.x;
            v[4 * q + 1] = x.y;
            v[4 * q + 2] = x.z;
            v[4 * q + 3] = x.w;
          }
          if (e.gain) {
            const float4* g4 = reinterpret_cast<const float4*>(e.gain + n);
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              const float4 gg = g4[q];
              ss += v[4 * q] * v[4 * q] + v[4 * q + 1] * v[4 * q + 1] +
                    v[4 * q + 2] * v[4 * q + 2] + v[4 * q + 3] * v[4 * q + 3];
              v[4 * q] *= gg.x;
              v[4 * q + 1] *= gg.y;
              v[4 * q + 2] *= gg.z;
              v[4 * q + 3] *= gg.w;
            }
            store_bf16x32(e.a_out + off, v);
          }
        }
      }
      if (live && e.gain)
        e.ss_out[static_cast<size_t>(m) * (N / 128) + nt * (BN / 128) + gq] = ss;
    }
  } else if constexpr (EPI == kEpiSwiglu) {
    static_assert(BN == 256, "the SwiGLU tile is 128 gate + 128 up columns");
    const SwigluEpilogue& e = g.swiglu;
    const float r =
        live ? rms_row_scale(e.rs.ss + static_cast<size_t>(m) * e.rs.ss_parts, e.rs.ss_parts,
                             e.rs.inv_d, e.rs.eps)
             : 0.f;
    for (int jj = 0; jj < 4; ++jj) {
      float gv[32], uv[32];
      load_chunk<BN>(g, taddr, fx, jj, row, gv);
      load_chunk<BN>(g, taddr, fx, 4 + jj, row, uv);
      if (live) {
#pragma unroll
        for (int i = 0; i < 32; ++i) gv[i] = silu(r * gv[i]) * (r * uv[i]);
        store_bf16x32(e.act + static_cast<size_t>(m) * e.ffn + nt * 128 + jj * 32, gv);
      }
    }
  } else {
    const QkvEpilogue& e = g.qkv;
    const int half = e.head_dim / 2;
    const float r =
        live ? rms_row_scale(e.rs.ss + static_cast<size_t>(m) * e.rs.ss_parts, e.rs.ss_parts,
                             e.rs.inv_d, e.rs.eps)
             : 0.f;
    for (int hh = 0; hh < BN / 128; ++hh) {
      const int c0 = nt * BN + hh * 128;
      if (c0 >= e.q_width + e.kv_width) {
        uint16_t* dst = e.v_cache + static_cast<size_t>(e.start_pos + m) * e.kv_width +
                        (c0 - e.q_width - e.kv_width);
        for (int jj = 0; jj < 4; ++jj) {
          float v[32];
          load_chunk<BN>(g, taddr, fx, hh * 4 + jj, row, v);
          if (live) {
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] *= r;
            store_bf16x32(dst + jj * 32, v);
          }
        }
      } else {
        uint16_t* dst = c0 < e.q_width
                            ? e.q + static_cast<size_t>(m) * e.q_width + c0
                            : e.k_cache + static_cast<size_t>(e.start_pos + m) * e.kv_width +
                                  (c0 - e.q_width);
        const float2* cs = e.rope + static_cast<size_t>(m) * half;
        for (int p = 0; p < 2; ++p) {
          // head_dim 128: one head per 128 columns, pairs (chunk 0, 2) and (1, 3);
          // head_dim 64: two heads, pairs (0, 1) and (2, 3).
          const int ja = (e.head_dim == 128) ? p : 2 * p;
          const int jb = ja + half / 32;
          const int i0 = (e.head_dim == 128) ? p * 32 : 0;
          float va[32], vb[32];
          load_chunk<BN>(g, taddr, fx, hh * 4 + ja, row, va);
          load_chunk<BN>(g, taddr, fx, hh * 4 + jb, row, vb);
          if (live) {
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const float2 sc = cs[i0 + i];
              const float u = r * va[i], w = r * vb[i];
              va[i] = u * sc.x - w * sc.y;
              vb[i] = u * sc.y + w * sc.x;
            }
            store_bf16x32(dst + ja * 32, va);
            store_bf16x32(dst + jb * 32, vb);
          }
        }
      }
    }
  }
}

template <int BN, int EPI>
__global__ void __launch_bounds__(192, 1)
    gemm_kernel(const __grid_constant__ GemmMaps maps, const __grid_constant__ GemmArgs g) {
  using namespace sm100;
  using C = Cfg<BN>;
  constexpr int S = C::kStages;
  constexpr uint32_t kIdesc = idesc_bf16_f32(BM, BN);

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

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cta = blockIdx.x;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(bar_full(s), 1);
      mbar_init(bar_empty(s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(bar_tfull(a), 1);
      mbar_init(bar_tempty(a), 128);
    }
    mbar_init(bar_drain, 1);
    *abort_flag = 0;
    mbar_init_fence();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_map(&maps.a);
    tma_prefetch_map(&maps.b[0]);
    tma_prefetch_map(&maps.b[1]);
    tma_prefetch_map(&maps.b[2]);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(misc), C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = misc[0];

  // Everything above overlaps the previous kernel when launched with
  // programmatic stream serialization; the inputs are only read below.
  grid_dep_wait();
  grid_dep_launch();

  const int it0 = seg_begin(g, cta), it1 = seg_begin(g, cta + 1);
  int issued = 0;  // producer: k-block loads issued
  int consumed = 0;

  if (warp == 0) {
    if (lane == 0) {
      const uint64_t pol_w = policy_evict_first(), pol_a = policy_evict_last();
      SegIter si{it0, it1, g.kb};
      int tile, k0, k1;
      bool ok = true;
      while (ok && si.next(tile, k0, k1)) {
        const int mt = tile % g.tiles_m, nt = tile / g.tiles_m;
        for (int kb = k0; kb < k1; ++kb) {
          const int s = issued % S;
          if (!mbar_wait(bar_empty(s), ((issued / S) & 1) ^ 1, abort_flag, g.status)) {
            ok = false;
            break;
          }
          const uint32_t dst = sbase + s * C::kStage;
          mbar_arrive_expect_tx(bar_full(s), C::kStage);
          tma_load_2d(dst, &maps.a, bar_full(s), kb * BK, mt * BM, pol_a);
#pragma unroll
          for (int h = 0; h < BN / 128; ++h) {
            int mi, row;
            b_source<BN>(g, nt, h, mi, row);
            tma_load_2d(dst + C::kABytes + h * 16384u, &maps.b[mi], bar_full(s), kb * BK, row,
                        pol_w);
          }
          ++issued;
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
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
          const uint32_t a_addr = sbase + s * C::kStage;
          const uint64_t ad = smem_desc_sw128(a_addr);
          const uint64_t bd = smem_desc_sw128(a_addr + C::kABytes);
#pragma unroll
          for (int k = 0; k < BK / 16; ++k)
            umma_bf16(d_tmem, ad + 2u * k, bd + 2u * k, kIdesc, (kb > k0 || k > 0) ? 1u : 0u);
          umma_commit(bar_empty(s));
          ++consumed;
        }
        if (!ok) break;
        umma_commit(bar_tfull(ab));
        ++sg;
      }
      // Every MMA this thread issued has completed before TMEM is released.
      umma_commit(bar_drain);
      int dummy_abort = 0;
      mbar_wait(bar_drain, 0, &dummy_abort, g.status);
    }
  } else {
    const int lane_grp = warp & 3;  // this warp's TMEM lanes: 32*lane_grp ..
    const int row = lane_grp * 32 + lane;
    SegIter si{it0, it1, g.kb};
    int tile, k0, k1, sg = 0;
    while (si.next(tile, k0, k1)) {
      const int ab = sg & 1;
      if (!mbar_wait(bar_tfull(ab), (sg >> 1) & 1, abort_flag, g.status)) break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(lane_grp * 32) << 16) + ab * BN;
      const int mt = tile % g.tiles_m, nt = tile / g.tiles_m;
      const int m = mt * BM + row;
      Fixup fx{false, 0, 0, cta, tile};
      bool run = true;
      if (!(k0 == 0 && k1 == g.kb)) {
        const int slot = (it0 / g.kb == tile) ? 0 : 1;
        float4* mine =
            reinterpret_cast<float4*>(g.partials) + static_cast<size_t>(cta * 2 + slot) * (BM * BN / 4);
        for (int j = 0; j < BN / 32; ++j) {
          float v[32];
          tmem_load32(taddr + j * 32, v);
#pragma unroll
          for (int q = 0; q < 8; ++q)
            __stcg(mine + (j * 8 + q) * BM + row,
                   make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]));
        }
        __threadfence();
        named_bar_sync(1, 128);
        if (threadIdx.x == 64) misc[1] = atomicAdd(&g.counters[tile], 1u);
        named_bar_sync(1, 128);
        const int arrived = static_cast<int>(misc[1]);
        const int cf = cta_of_iter(g, tile * g.kb), cl = cta_of_iter(g, tile * g.kb + g.kb - 1);
        if (arrived == cl - cf) {
          __threadfence();
          fx = Fixup{true, cf, cl, cta, tile};
        } else {
          run = false;
        }
      }
      if (run) {
        run_epilogue<BN, EPI>(g, taddr, fx, m, nt, row);
        if (fx.active && threadIdx.x == 64) g.counters[tile] = 0;
      }
      tc_fence_before();
      mbar_arrive(bar_tempty(ab));
      ++sg;
    }
  }

  // On a timeout the producer may have loads in flight: let them land
  // (bounded) before the CTA's shared memory is released.
  if (warp == 0 && lane == 0 && *abort_flag) {
    int dummy_abort = 0;
    for (int i = max(0, issued - S); i < issued; ++i)
      mbar_wait(bar_full(i % S), (i / S) & 1, &dummy_abort, g.status);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, C::kTmemCols);
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
  bool operator==(const TmapKey& o) const { return p == o.p && inner == o.inner && outer == o.outer; }
};
struct TmapKeyHash {
  size_t operator()(const TmapKey& k) const {
    return std::hash<const void*>()(k.p) ^ (k.inner * 0x9E3779B97F4A7C15ull) ^ (k.outer << 20);
  }
};
struct TmapCache {
  std::mutex mu;
  std::unordered_map<TmapKey, CUtensorMap, TmapKeyHash> maps;
};

TmapCache* tmap_cache_create() { return new TmapCache(); }
void tmap_cache_destroy(TmapCache* c) { delete c; }

namespace {

// bf16 matrix [outer rows, inner columns], box of 64 columns x 128 rows, 128-byte swizzle.
pds_status get_map(TcContext& c, CUtensorMap* out, const void* p, uint64_t inner, uint64_t outer,
                   std::string* err) {
  TmapKey key{p, inner, outer};
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
  const cuuint64_t strides[1] = {inner * 2};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(BK), 128};
  const cuuint32_t es[2] = {1, 1};
  CUresult r = fn(out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(p), dims, strides, box,
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

void make_schedule(GemmArgs& g, const TcContext& c, int M, int tiles_n, int K) {
  g.M = M;
  g.K = K;
  g.tiles_m = (M + BM - 1) / BM;
  g.tiles_n = tiles_n;
  g.kb = K / BK;
  g.total = g.tiles_m * g.tiles_n * g.kb;
  int grid = std::min(c.num_sms > 0 ? c.num_sms : 148, kGemmMaxGrid);
  grid = std::min(grid, std::max(1, g.total / kMinItersPerCta));
  g.grid = grid;
}

template <int BN, int EPI>
pds_status launch(TcContext& c, const GemmMaps& maps, GemmArgs& g, cudaStream_t st,
                  std::string* err) {
  using Cf = Cfg<BN>;
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(gemm_kernel<BN, EPI>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    static_cast<int>(Cf::kSmem));
  });
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
  cfg.gridDim = dim3(g.grid);
  cfg.blockDim = dim3(192);
  cfg.dynamicSmemBytes = Cf::kSmem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = c.pdl ? 1 : 0;
  cudaError_t ce = cudaLaunchKernelEx(&cfg, gemm_kernel<BN, EPI>, maps, g);
  if (ce != cudaSuccess) {
    *err = std::string("gemm launch: ") + cudaGetErrorString(ce);
    return PDS_ELAUNCH;
  }
  return PDS_OK;
}

}  // namespace

size_t tc_gemm_scratch_bytes(int M, int max_tiles_n) {
  const size_t part_bytes = static_cast<size_t>(kGemmMaxGrid) * 2 * BM * 256 * sizeof(float);
  const size_t tiles = static_cast<size_t>((M + BM - 1) / BM) * max_tiles_n;
  return part_bytes + ((tiles * 4 + 255) / 256) * 256;
}

pds_status tc_gemm_plain(TcContext& c, const uint16_t* A, const uint16_t* W, float* Cout, int M,
                         int N, int K, cudaStream_t st, std::string* err) {
  GemmMaps maps;
  pds_status rc;
  if ((rc = get_map(c, &maps.a, A, K, M, err)) != PDS_OK) return rc;
  if ((rc = get_map(c, &maps.b[0], W, K, N, err)) != PDS_OK) return rc;
  maps.b[1] = maps.b[0];
  maps.b[2] = maps.b[0];
  GemmArgs g{};
  g.wrows0 = N;
  g.wrows1 = 0;
  g.c_out = Cout;
  g.ldc = N;
  if (N % 256 == 0) {
    make_schedule(g, c, M, N / 256, K);
    return launch<256, kEpiPlain>(c, maps, g, st, err);
  }
  make_schedule(g, c, M, N / 128, K);
  return launch<128, kEpiPlain>(c, maps, g, st, err);
}

pds_status tc_gemm_resid(TcContext& c, const uint16_t* A, const uint16_t* W, int M, int N, int K,
                         const ResidEpilogue& e, cudaStream_t st, std::string* err) {
  GemmMaps maps;
  pds_status rc;
  if ((rc = get_map(c, &maps.a, A, K, M, err)) != PDS_OK) return rc;
  if ((rc = get_map(c, &maps.b[0], W, K, N, err)) != PDS_OK) return rc;
  maps.b[1] = maps.b[0];
  maps.b[2] = maps.b[0];
  GemmArgs g{};
  g.wrows0 = N;
  g.resid = e;
  g.resid_n = N;
  if (N % 256 == 0) {
    make_schedule(g, c, M, N / 256, K);
    return launch<256, kEpiResid>(c, maps, g, st, err);
  }
  make_schedule(g, c, M, N / 128, K);
  return launch<128, kEpiResid>(c, maps, g, st, err);
}

pds_status tc_gemm_swiglu(TcContext& c, const uint16_t* A, const WeightRows& W, int M, int K,
                          const SwigluEpilogue& e, cudaStream_t st, std::string* err) {
  GemmMaps maps;
  pds_status rc;
  if ((rc = get_map(c, &maps.a, A, K, M, err)) != PDS_OK) return rc;
  if ((rc = get_map(c, &maps.b[0], W.w[0], K, W.rows[0], err)) != PDS_OK) return rc;
  if ((rc = get_map(c, &maps.b[1], W.w[1], K, W.rows[1], err)) != PDS_OK) return rc;
  maps.b[2] = maps.b[0];
  GemmArgs g{};
  g.pair_mode = 1;
  g.swiglu = e;
  make_schedule(g, c, M, e.ffn / 128, K);
  return launch<256, kEpiSwiglu>(c, maps, g, st, err);
}

pds_status tc_gemm_qkv(TcContext& c, const uint16_t* A, const WeightRows& W, int M, int K,
                       const QkvEpilogue& e, cudaStream_t st, std::string* err) {
  GemmMaps maps;
  pds_status rc;
  if ((rc = get_map(c, &maps.a, A, K, M, err)) != PDS_OK) return rc;
  for (int i = 0; i < 3; ++i)
    if ((rc = get_map(c, &maps.b[i], W.w[i], K, W.rows[i], err)) != PDS_OK) return rc;
  GemmArgs g{};
  g.wrows0 = W.rows[0];
  g.wrows1 = W.rows[1];
  g.qkv = e;
  const int N = W.rows[0] + W.rows[1] + W.rows[2];
  if (N % 256 == 0) {
    make_schedule(g, c, M, N / 256, K);
    return launch<256, kEpiQkv>(c, maps, g, st, err);
  }
  make_schedule(g, c, M, N / 128, K);
  return launch<128, kEpiQkv>(c, maps, g, st, err);
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
  cudaError_t ce = cudaMemsetAsync(counters, 0, tiles * 4, st);
  if (ce != cudaSuccess) {
    *err = std::string("static scratch counter reset: ") + cudaGetErrorString(ce);
    return PDS_ELAUNCH;
  }
  TcContext c{};
  c.num_sms = num_sms;
  GemmMaps maps;
  if ((rc = get_map(c, &maps.a, A, K, M, err)) != PDS_OK) return rc;
  if ((rc = get_map(c, &maps.b[0], W, K, N, err)) != PDS_OK) return rc;
  maps.b[1] = maps.b[0];
  maps.b[2] = maps.b[0];
  GemmArgs g{};
  g.wrows0 = N;
  g.c_out = Cout;
  g.ldc = N;
  make_schedule(g, c, M, N / kNoAllocBN, K);
  g.grid = std::min(g.grid, grid_cap);
  g.status = status;
  g.partials = partials;
  g.counters = counters;

  using Cf = Cfg<kNoAllocBN>;
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(gemm_kernel<kNoAllocBN, kEpiPlain>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    static_cast<int>(Cf::kSmem));
  });
  if (attr_err != cudaSuccess) {
    *err = std::string("gemm shared-memory attribute: ") + cudaGetErrorString(attr_err);
    return PDS_ELAUNCH;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(g.grid);
  cfg.blockDim = dim3(192);
  cfg.dynamicSmemBytes = Cf::kSmem;
  cfg.stream = st;
  ce = cudaLaunchKernelEx(&cfg, gemm_kernel<kNoAllocBN, kEpiPlain>, maps, g);
  if (ce != cudaSuccess) {
    *err = std::string("gemm launch: ") + cudaGetErrorString(ce);
    return PDS_ELAUNCH;
  }
  return PDS_OK;
}

}  // namespace pds
