// pod_k1_lt.cu — K1 instantiations with a logits transform (soft cap or
// ALiBi) on both halves, fp16/bf16 x head_dim 64/128.
#include "pod_k1.h"
#include "pod_kernels.cuh"

cudaError_t pod_k1_lt(const PodParams& P, int dtype, cudaStream_t stream) {
  const bool cap = P.lt == POD_LT_SOFTCAP;
  if (P.d == 128) {
    if (dtype == 1)
      return cap ? launch_pod<__nv_bfloat16, 128, false, POD_LT_SOFTCAP, false>(P, stream)
                 : launch_pod<__nv_bfloat16, 128, false, POD_LT_ALIBI, false>(P, stream);
    return cap ? launch_pod<__half, 128, false, POD_LT_SOFTCAP, false>(P, stream)
               : launch_pod<__half, 128, false, POD_LT_ALIBI, false>(P, stream);
  }
  if (dtype == 1)
    return cap ? launch_pod<__nv_bfloat16, 64, false, POD_LT_SOFTCAP, false>(P, stream)
               : launch_pod<__nv_bfloat16, 64, false, POD_LT_ALIBI, false>(P, stream);
  return cap ? launch_pod<__half, 64, false, POD_LT_SOFTCAP, false>(P, stream)
             : launch_pod<__half, 64, false, POD_LT_ALIBI, false>(P, stream);
}
