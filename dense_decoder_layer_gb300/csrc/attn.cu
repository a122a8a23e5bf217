// GQA causal attention of the new rows over the cache prefix plus the new
// rows (frink-models 0.29.0 src/decoder/cuda_prefill.rs, PrefillParams:
// prefix_k / prefix_v are the cache's first start_pos rows; attn_scale =
// 1/sqrt(head_dim); no softcap, no window).
//
// Flash-style: one CTA per (64 query rows, query head), 4 warps of 16 rows.
// K/V tiles of 64 keys are staged in shared memory (double-buffered async
// copies, XOR-swizzled 16-byte chunks so ldmatrix is conflict-free);
// S = Q.K^T and O += P.V run on the tensor cores (bf16 in, fp32 out); the
// softmax is online, in base 2, with the running max and sum per row kept
// by the 4 threads that own the row.  Key tiles past the CTA's last
// position are never loaded; tiles that reach past a row's position are
// masked.  Query row b sits at position start_pos + b and reads kv head
// h / (H / Hkv).
#include <cuda_runtime.h>

#include "common.cuh"
#include "kernels.h"
#include "tc.h"

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

template <int HD>
__global__ void __launch_bounds__(128) flash_attn_kernel(const uint16_t* __restrict__ q,
                                                         const uint16_t* __restrict__ k,
                                                         const uint16_t* __restrict__ v,
                                                         uint16_t* __restrict__ o, int B, int s,
                                                         int H, int Hkv, float scale_log2) {
  constexpr int CH = HD / 8;  // 16-byte chunks per row
  extern __shared__ __align__(128) uint16_t smem[];
  uint16_t* sQ = smem;
  uint16_t* sK = sQ + kBM * HD;
  uint16_t* sV = sK + 2 * kBN * HD;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int qt = gridDim.x - 1 - blockIdx.x;  // longest tiles first
  const int h = blockIdx.y, g = h / (H / Hkv);
  const int b0 = qt * kBM;
  const int T = s + B;
  const int last_row = min(b0 + kBM, B) - 1;
  const int kv_end = s + last_row + 1;
  const int nkt = (kv_end + kBN - 1) / kBN;

  for (int i = tid; i < kBM * CH; i += 128) {
    const int r = i / CH, c = i % CH, b = b0 + r;
    cp_async16(smem_addr(sQ + swz<HD>(r, c)),
               q + (static_cast<size_t>(min(b, B - 1)) * H + h) * HD + c * 8, b < B ? 16 : 0);
  }
  auto load_kv = [&](int kt, int buf) {
    uint16_t* dk = sK + buf * kBN * HD;
    uint16_t* dv = sV + buf * kBN * HD;
    for (int i = tid; i < kBN * CH; i += 128) {
      const int r = i / CH, c = i % CH, j = kt * kBN + r;
      const size_t off = (static_cast<size_t>(min(j, T - 1)) * Hkv + g) * HD + c * 8;
      const int n = j < T ? 16 : 0;
      cp_async16(smem_addr(dk + swz<HD>(r, c)), k + off, n);
      cp_async16(smem_addr(dv + swz<HD>(r, c)), v + off, n);
    }
  };
  load_kv(0, 0);
  cp_async_commit();

  uint32_t qf[HD / 16][4];
  float oacc[HD / 8][4];
#pragma unroll
  for (int i = 0; i < HD / 8; ++i) oacc[i][0] = oacc[i][1] = oacc[i][2] = oacc[i][3] = 0.f;
  float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
  const int r_lo = warp * 16 + (lane >> 2);
  const int pos0 = s + b0 + r_lo, pos1 = pos0 + 8;
  const int warp_min_pos = s + b0 + warp * 16;

  for (int kt = 0; kt < nkt; ++kt) {
    const int buf = kt & 1;
    if (kt + 1 < nkt) load_kv(kt + 1, buf ^ 1);
    cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();
    if (kt == 0) {
#pragma unroll
      for (int kk = 0; kk < HD / 16; ++kk) {
        const int row = warp * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
        ldsm_x4(qf[kk], smem_addr(sQ + swz<HD>(row, kk * 2 + (lane >> 4))));
      }
    }
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
    __syncthreads();
  }

  float l0 = l_run[0], l1 = l_run[1];
  l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
  const float inv0 = 1.f / l0, inv1 = 1.f / l1;
  const int row0 = b0 + r_lo, row1 = row0 + 8;
#pragma unroll
  for (int nb = 0; nb < HD / 8; ++nb) {
    const int col = h * HD + nb * 8 + 2 * (lane & 3);
    if (row0 < B)
      *reinterpret_cast<uint32_t*>(o + static_cast<size_t>(row0) * H * HD + col) =
          pack_bf16x2(oacc[nb][0] * inv0, oacc[nb][1] * inv0);
    if (row1 < B)
      *reinterpret_cast<uint32_t*>(o + static_cast<size_t>(row1) * H * HD + col) =
          pack_bf16x2(oacc[nb][2] * inv1, oacc[nb][3] * inv1);
  }
}

template <int HD>
cudaError_t launch_flash(const uint16_t* q, const uint16_t* k, const uint16_t* v, uint16_t* o,
                         int B, int s, int H, int Hkv, cudaStream_t st) {
  constexpr size_t smem = static_cast<size_t>(kBM + 4 * kBN) * HD * sizeof(uint16_t);
  static cudaError_t attr = cudaFuncSetAttribute(
      flash_attn_kernel<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (attr != cudaSuccess) return attr;
  const float scale_log2 = 1.4426950408889634f / sqrtf(static_cast<float>(HD));
  dim3 grid((B + kBM - 1) / kBM, H);
  flash_attn_kernel<HD><<<grid, 128, smem, st>>>(q, k, v, o, B, s, H, Hkv, scale_log2);
  return cudaGetLastError();
}

}  // namespace

pds_status tc_attention(TcContext& c, const uint16_t* q, const uint16_t* k, const uint16_t* v,
                        uint16_t* o, int B, int start_pos, int H, int Hkv, int hd, cudaStream_t st,
                        std::string* err) {
  (void)c;
  cudaError_t ce = hd == 128 ? launch_flash<128>(q, k, v, o, B, start_pos, H, Hkv, st)
                             : launch_flash<64>(q, k, v, o, B, start_pos, H, Hkv, st);
  if (ce != cudaSuccess) {
    *err = std::string("attention launch: ") + cudaGetErrorString(ce);
    return PDS_ELAUNCH;
  }
  return PDS_OK;
}

}  // namespace pds
