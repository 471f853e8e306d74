// pod_launch.h — host entry into the kernels (pod_launch.cu).
#pragma once
#include <cuda_runtime.h>

#include "pod_plan.h"

// Launch the fused POD kernel and, when the plan split any KV range, the
// PDL-chained merge kernel. dtype: 0 = fp16, 1 = bf16.
cudaError_t pod_launch(const PodParams& P, int dtype, cudaStream_t stream);

// Dynamic shared memory of the fused kernel for head_dim d (rope: the RoPE kernel).
int pod_kernel_smem_bytes(int d, int rope);
