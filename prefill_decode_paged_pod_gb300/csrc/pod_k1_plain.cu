// pod_k1_plain.cu — K1 instantiations without a logits transform or RoPE:
// fp16/bf16 x head_dim 64/128/256, and the FP8 (E4M3) decode cache at 128.
#include "pod_k1.h"
#include "pod_kernels.cuh"

cudaError_t pod_k1_plain(const PodParams& P, int dtype, cudaStream_t stream) {
  if (P.d == 256)   // one CTA per SM: O takes 256 TMEM columns
    return dtype == 1 ? launch_pod<__nv_bfloat16, 256, false, POD_LT_NONE, false>(P, stream)
                      : launch_pod<__half, 256, false, POD_LT_NONE, false>(P, stream);
  if (P.d == 128) {
    if (dtype == 1)
      return P.d_fp8 ? launch_pod<__nv_bfloat16, 128, true, POD_LT_NONE, false>(P, stream)
                     : launch_pod<__nv_bfloat16, 128, false, POD_LT_NONE, false>(P, stream);
    return P.d_fp8 ? launch_pod<__half, 128, true, POD_LT_NONE, false>(P, stream)
                   : launch_pod<__half, 128, false, POD_LT_NONE, false>(P, stream);
  }
  return dtype == 1 ? launch_pod<__nv_bfloat16, 64, false, POD_LT_NONE, false>(P, stream)
                    : launch_pod<__half, 64, false, POD_LT_NONE, false>(P, stream);
}

int pod_k1_smem_plain(int d) {
  return d == 256 ? smem_bytes<256, false>() : d == 128 ? smem_bytes<128, false>() : smem_bytes<64, false>();
}
