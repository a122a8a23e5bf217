// GQA causal attention of the new rows over the cache prefix plus the new
// rows (frink-models 0.29.0 src/decoder/cuda_prefill.rs, PrefillParams:
// prefix_k / prefix_v are the cache's first start_pos rows; attn_scale =
// 1/sqrt(head_dim); no softcap, no window).
#include <cuda_runtime.h>

#include "kernels.h"
#include "tc.h"

namespace pds {

pds_status tc_attention(TcContext& c, const uint16_t* q, const uint16_t* k, const uint16_t* v,
                        uint16_t* o, int B, int start_pos, int H, int Hkv, int hd, cudaStream_t st,
                        std::string* err) {
  (void)c;
  launch_attention_naive(q, k, v, o, B, start_pos, H, Hkv, hd, st);
  cudaError_t ce = cudaGetLastError();
  if (ce != cudaSuccess) {
    *err = std::string("attention launch: ") + cudaGetErrorString(ce);
    return PDS_ELAUNCH;
  }
  return PDS_OK;
}

}  // namespace pds
