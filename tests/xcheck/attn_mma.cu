// TEST-ONLY cross-check (built into its own library, libpds_xcheck.so,
// never into the product's libpds.so): a second, independent GPU
// implementation of the stack's attention on the warp-level mma.sync tensor
// path, for comparing the tcgen05 kernel against on the same inputs.
//
// GQA causal attention of the new rows over the cache prefix plus the new
// rows (frink-models 0.29.0 src/decoder/cuda_prefill.rs, PrefillParams:
// prefix_k / prefix_v are the cache's first start_pos rows; attn_scale =
// 1/sqrt(head_dim); no softcap, no window).
//
// Flash-style: one CTA per (64 query rows, query head), two halves of 4
// warps (16 rows each) that split the key tiles between them.  K/V tiles of
// 64 keys are staged in shared memory (double-buffered async copies per
// half, XOR-swizzled 16-byte chunks so ldmatrix is conflict-free);
// S = Q.K^T and O += P.V run on the tensor cores (bf16 in, fp32 out); the
// softmax is online, in base 2, with the running max and sum per row kept
// by the 4 threads that own the row.  Key tiles past the CTA's last
// position are never loaded; tiles that reach past a row's position are
// masked.  Query row b sits at position start_pos + b and reads kv head
// h / (H / Hkv).
#include <cuda_runtime.h>

#include <math.h>
#include <stdint.h>

#include "common.cuh"

namespace pds {
namespace {

constexpr int kBM = 64;  // query rows per CTA
constexpr int kBN = 64;  // keys per tile

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
               "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void named_barrier(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

// D (16x8 fp32) += A (16x16 bf16, row) * B (16x8 bf16, col)
__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Element offset of the 16-byte chunk `chunk` of row `row` in a [rows][HD] tile.
template <int HD>
__device__ __forceinline__ int swz(int row, int chunk) {
  return row * HD + ((chunk ^ (row & 7)) << 3);
}

// The two halves of a CTA (warps 0-3 and 4-7) take alternate key tiles of
// the same 64 query rows, each with its own double-buffered K/V tiles and
// its own running max, sum and output; at the end the second half hands its
// state to the first through shared memory and the first merges the two.
template <int HD>
__global__ void __launch_bounds__(256) flash_attn_kernel(const uint16_t* __restrict__ q,
                                                         const uint16_t* __restrict__ k,
                                                         const uint16_t* __restrict__ v,
                                                         uint16_t* __restrict__ o, int B, int s,
                                                         int H, int Hkv, float scale_log2) {
  constexpr int CH = HD / 8;  // 16-byte chunks per row
  extern __shared__ __align__(128) uint16_t smem[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int kh = warp >> 2;   // which half: key tiles kh, kh + 2, ...
  const int wq = warp & 3;    // which 16 query rows
  const int htid = tid & 127;
  uint16_t* sQ = smem;
  uint16_t* sK = sQ + kBM * HD + kh * (4 * kBN * HD);  // this half's 2 K then 2 V tiles
  uint16_t* sV = sK + 2 * kBN * HD;

  const int qt = gridDim.y - 1 - blockIdx.y;  // longest row tiles first, over all heads
  const int h = blockIdx.x, g = h / (H / Hkv);
  const int b0 = qt * kBM;
  const int T = s + B;
  const int last_row = min(b0 + kBM, B) - 1;
  const int kv_end = s + last_row + 1;
  const int nkt = (kv_end + kBN - 1) / kBN;
  const int nmine = nkt > kh ? (nkt - kh + 1) / 2 : 0;

  // q, k and v are the previous kernel's output
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");

  for (int i = tid; i < kBM * CH; i += 256) {
    const int r = i / CH, c = i % CH, b = b0 + r;
    cp_async16(smem_addr(sQ + swz<HD>(r, c)),
               q + (static_cast<size_t>(min(b, B - 1)) * H + h) * HD + c * 8, b < B ? 16 : 0);
  }
  cp_async_commit();
  auto load_kv = [&](int kt, int buf) {
    uint16_t* dk = sK + buf * kBN * HD;
    uint16_t* dv = sV + buf * kBN * HD;
    for (int i = htid; i < kBN * CH; i += 128) {
      const int r = i / CH, c = i % CH, j = kt * kBN + r;
      const size_t off = (static_cast<size_t>(min(j, T - 1)) * Hkv + g) * HD + c * 8;
      const int n = j < T ? 16 : 0;
      cp_async16(smem_addr(dk + swz<HD>(r, c)), k + off, n);
      cp_async16(smem_addr(dv + swz<HD>(r, c)), v + off, n);
    }
  };
  if (nmine > 0) load_kv(kh, 0);
  cp_async_commit();
  cp_async_wait<1>();  // this thread's part of Q
  __syncthreads();     // everyone's

  uint32_t qf[HD / 16][4];
#pragma unroll
  for (int kk = 0; kk < HD / 16; ++kk) {
    const int row = wq * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
    ldsm_x4(qf[kk], smem_addr(sQ + swz<HD>(row, kk * 2 + (lane >> 4))));
  }
  float oacc[HD / 8][4];
#pragma unroll
  for (int i = 0; i < HD / 8; ++i) oacc[i][0] = oacc[i][1] = oacc[i][2] = oacc[i][3] = 0.f;
  float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
  const int r_lo = wq * 16 + (lane >> 2);
  const int pos0 = s + b0 + r_lo, pos1 = pos0 + 8;
  const int warp_min_pos = s + b0 + wq * 16;

  for (int it = 0; it < nmine; ++it) {
    const int kt = kh + 2 * it;
    const int buf = it & 1;
    if (it + 1 < nmine) load_kv(kt + 2, buf ^ 1);
    cp_async_commit();
    cp_async_wait<1>();
    named_barrier(1 + kh, 128);
    const uint16_t* tK = sK + buf * kBN * HD;
    const uint16_t* tV = sV + buf * kBN * HD;

    float sacc[kBN / 8][4];
#pragma unroll
    for (int i = 0; i < kBN / 8; ++i) sacc[i][0] = sacc[i][1] = sacc[i][2] = sacc[i][3] = 0.f;
#pragma unroll
    for (int kk = 0; kk < HD / 16; ++kk) {
#pragma unroll
      for (int nb = 0; nb < kBN / 8; nb += 2) {
        uint32_t b[4];
        const int key = nb * 8 + (lane & 7) + (lane >> 4) * 8;
        ldsm_x4(b, smem_addr(tK + swz<HD>(key, kk * 2 + ((lane >> 3) & 1))));
        mma_bf16(sacc[nb], qf[kk], b[0], b[1]);
        mma_bf16(sacc[nb + 1], qf[kk], b[2], b[3]);
      }
    }

    const int kbase = kt * kBN;
    const bool mask = kbase + kBN - 1 > warp_min_pos;
    float mx0 = m_run[0], mx1 = m_run[1];
#pragma unroll
    for (int nb = 0; nb < kBN / 8; ++nb) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float t = sacc[nb][e] * scale_log2;
        if (mask) {
          const int key = kbase + nb * 8 + 2 * (lane & 3) + (e & 1);
          if (key > (e < 2 ? pos0 : pos1)) t = -INFINITY;
        }
        sacc[nb][e] = t;
      }
      mx0 = fmaxf(mx0, fmaxf(sacc[nb][0], sacc[nb][1]));
      mx1 = fmaxf(mx1, fmaxf(sacc[nb][2], sacc[nb][3]));
    }
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
    const float ref0 = mx0 == -INFINITY ? 0.f : mx0;
    const float ref1 = mx1 == -INFINITY ? 0.f : mx1;
    const float al0 = exp2f(m_run[0] - ref0), al1 = exp2f(m_run[1] - ref1);
    m_run[0] = mx0;
    m_run[1] = mx1;

    uint32_t pf[kBN / 16][4];
    float sum0 = 0.f, sum1 = 0.f;
#pragma unroll
    for (int nb = 0; nb < kBN / 8; ++nb) {
      const float p0 = exp2f(sacc[nb][0] - ref0), p1 = exp2f(sacc[nb][1] - ref0);
      const float p2 = exp2f(sacc[nb][2] - ref1), p3 = exp2f(sacc[nb][3] - ref1);
      sum0 += p0 + p1;
      sum1 += p2 + p3;
      pf[nb >> 1][(nb & 1) * 2 + 0] = pack_bf16x2(p0, p1);
      pf[nb >> 1][(nb & 1) * 2 + 1] = pack_bf16x2(p2, p3);
    }
    l_run[0] = l_run[0] * al0 + sum0;
    l_run[1] = l_run[1] * al1 + sum1;
#pragma unroll
    for (int nb = 0; nb < HD / 8; ++nb) {
      oacc[nb][0] *= al0;
      oacc[nb][1] *= al0;
      oacc[nb][2] *= al1;
      oacc[nb][3] *= al1;
    }
#pragma unroll
    for (int kk = 0; kk < kBN / 16; ++kk) {
#pragma unroll
      for (int nb = 0; nb < HD / 8; nb += 2) {
        uint32_t b[4];
        const int key = kk * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
        ldsm_x4_t(b, smem_addr(tV + swz<HD>(key, nb + (lane >> 4))));
        mma_bf16(oacc[nb], pf[kk], b[0], b[1]);
        mma_bf16(oacc[nb + 1], pf[kk], b[2], b[3]);
      }
    }
    named_barrier(1 + kh, 128);  // the tile is consumed before its buffer is refilled
  }

  // Merge: the second half's state through shared memory (the K/V tiles'
  // space, free now), in the fragment layout, one word per lane.
  cp_async_wait<0>();
  __syncthreads();
  constexpr int kWords = HD / 2 + 4;  // oacc, then m, l per fragment row
  float* xch = reinterpret_cast<float*>(smem + kBM * HD) + wq * (kWords * 32);
  if (kh == 1) {
#pragma unroll
    for (int nb = 0; nb < HD / 8; ++nb)
#pragma unroll
      for (int e = 0; e < 4; ++e) xch[(nb * 4 + e) * 32 + lane] = oacc[nb][e];
    xch[(HD / 2 + 0) * 32 + lane] = m_run[0];
    xch[(HD / 2 + 1) * 32 + lane] = m_run[1];
    xch[(HD / 2 + 2) * 32 + lane] = l_run[0];
    xch[(HD / 2 + 3) * 32 + lane] = l_run[1];
  }
  __syncthreads();
  if (kh == 1) return;
  const float m1a = xch[(HD / 2 + 0) * 32 + lane], m1b = xch[(HD / 2 + 1) * 32 + lane];
  const float m0 = fmaxf(m_run[0], m1a), m1 = fmaxf(m_run[1], m1b);
  // the first half always sees key 0, so m0 and m1 are finite
  const float a00 = exp2f(m_run[0] - m0), a10 = exp2f(m1a - m0);
  const float a01 = exp2f(m_run[1] - m1), a11 = exp2f(m1b - m1);
  float l0 = l_run[0] * a00 + xch[(HD / 2 + 2) * 32 + lane] * a10;
  float l1 = l_run[1] * a01 + xch[(HD / 2 + 3) * 32 + lane] * a11;
  l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
  const float inv0 = 1.f / l0, inv1 = 1.f / l1;
  const int row0 = b0 + r_lo, row1 = row0 + 8;
#pragma unroll
  for (int nb = 0; nb < HD / 8; ++nb) {
    const float o0 = oacc[nb][0] * a00 + xch[(nb * 4 + 0) * 32 + lane] * a10;
    const float o1 = oacc[nb][1] * a00 + xch[(nb * 4 + 1) * 32 + lane] * a10;
    const float o2 = oacc[nb][2] * a01 + xch[(nb * 4 + 2) * 32 + lane] * a11;
    const float o3 = oacc[nb][3] * a01 + xch[(nb * 4 + 3) * 32 + lane] * a11;
    const int col = h * HD + nb * 8 + 2 * (lane & 3);
    if (row0 < B)
      *reinterpret_cast<uint32_t*>(o + static_cast<size_t>(row0) * H * HD + col) =
          pack_bf16x2(o0 * inv0, o1 * inv0);
    if (row1 < B)
      *reinterpret_cast<uint32_t*>(o + static_cast<size_t>(row1) * H * HD + col) =
          pack_bf16x2(o2 * inv1, o3 * inv1);
  }
}

template <int HD>
cudaError_t launch_flash(const uint16_t* q, const uint16_t* k, const uint16_t* v, uint16_t* o,
                         int B, int s, int H, int Hkv, bool pdl, cudaStream_t st) {
  constexpr size_t smem = static_cast<size_t>(kBM + 8 * kBN) * HD * sizeof(uint16_t);
  static_assert((HD / 2 + 4) * 32 * 4 * 4 <= 8 * kBN * HD * 2, "merge area");
  static cudaError_t attr = cudaFuncSetAttribute(
      flash_attn_kernel<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (attr != cudaSuccess) return attr;
  const float scale_log2 = 1.4426950408889634f / sqrtf(static_cast<float>(HD));
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(H, (B + kBM - 1) / kBM);
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute a[1];
  if (pdl) {
    a[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    a[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = a;
    cfg.numAttrs = 1;
  }
  return cudaLaunchKernelEx(&cfg, flash_attn_kernel<HD>, q, k, v, o, B, s, H, Hkv, scale_log2);
}

}  // namespace

}  // namespace pds

// 0 on success, else the cudaError_t of the failed launch.
extern "C" int pdsx_attention_mma(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                                  uint16_t* o, int32_t batch, int32_t start_pos, int32_t n_heads,
                                  int32_t n_kv_heads, int32_t head_dim, void* stream) {
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t ce = head_dim == 128
                       ? pds::launch_flash<128>(q, k, v, o, batch, start_pos, n_heads, n_kv_heads,
                                                false, st)
                       : pds::launch_flash<64>(q, k, v, o, batch, start_pos, n_heads, n_kv_heads,
                                               false, st);
  return static_cast<int>(ce);
}
