// pod_k1_rope.cu — K1 instantiations under ROPE_LLAMA (one CTA per SM; the
// soft cap is a run-time switch there), fp16/bf16 x head_dim 64/128.
#include "pod_k1.h"
#include "pod_kernels.cuh"

cudaError_t pod_k1_rope(const PodParams& P, int dtype, cudaStream_t stream) {
  if (P.d == 128)
    return dtype == 1 ? launch_pod<__nv_bfloat16, 128, false, POD_LT_NONE, true>(P, stream)
                      : launch_pod<__half, 128, false, POD_LT_NONE, true>(P, stream);
  return dtype == 1 ? launch_pod<__nv_bfloat16, 64, false, POD_LT_NONE, true>(P, stream)
                    : launch_pod<__half, 64, false, POD_LT_NONE, true>(P, stream);
}

int pod_k1_smem_rope(int d) { return d == 128 ? smem_bytes<128, true>() : smem_bytes<64, true>(); }
