// pod_k1.h — the K1 launchers, one per translation unit of instantiations.
#pragma once
#include <cuda_runtime.h>

#include "pod_plan.h"

cudaError_t pod_k1_plain(const PodParams& P, int dtype, cudaStream_t stream);
cudaError_t pod_k1_lt(const PodParams& P, int dtype, cudaStream_t stream);
cudaError_t pod_k1_rope(const PodParams& P, int dtype, cudaStream_t stream);
int pod_k1_smem_plain(int d);
int pod_k1_smem_rope(int d);
