// pod_launch.cu — the launch sequence of one POD run: K1 (the fused kernel,
// through the launcher of its variant) and, when the plan split any key
// range, K2 `pod_merge_kernel`.
//
// K2 merges the split partials of each row with base-2 LSE weights, adds the
// sink, writes out and LSE (flashinfer.cudnn page, "LSE 契约": base-2 LSE
// feeds a cascade merge). It is launched with programmatic dependent launch
// and waits on griddepcontrol.wait (POD walkthrough, "PDL"); K1 signals
// launch_dependents at its start.
#include <cuda_runtime.h>
#include <math.h>

#include "pod_device.cuh"
#include "pod_k1.h"
#include "pod_launch.h"
#include "pod_plan.h"

using namespace pod;

namespace {

template <typename T, int D>
__global__ void __launch_bounds__(256) pod_merge_kernel(const __grid_constant__ PodParams P) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int gw = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  // in CUDA-graph capacity mode the grid covers the capacity and the plan's
  // counts come from the workspace
  const int n_mrows = P.counts_in_ws ? P.status[POD_ST_NMROWS] : P.n_mrows;
  if (gw >= n_mrows) return;
  // merge group containing merge row gw
  int lo = 0, hi = (P.counts_in_ws ? P.status[POD_ST_NGROUPS] : P.n_groups) - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (P.mrow_ptr[mid] <= gw) lo = mid; else hi = mid - 1;
  }
  const int32_t* gr = P.mgroups + POD_REC * lo;
  const int half = gr[0], req = gr[1], g = gr[2], tok0 = gr[3], prow0 = gr[5], nsplit = gr[6],
            R = gr[7];
  const int r = gw - P.mrow_ptr[lo];
  const int tok = tok0 + r / P.G, head = g * P.G + r % P.G;
  float M = -INFINITY;
  for (int j = 0; j < nsplit; ++j) M = fmaxf(M, P.part_lse[prow0 + j * R + r]);
  const float Ms = (M == -INFINITY) ? 0.f : M;
  constexpr int PER = D / 32;
  float acc[PER];
#pragma unroll
  for (int i = 0; i < PER; ++i) acc[i] = 0.f;
  float wsum = 0.f;
  for (int j = 0; j < nsplit; ++j) {
    const int pr = prow0 + j * R + r;
    const float wgt = ex2(P.part_lse[pr] - Ms);
    wsum += wgt;
    const float* src = P.part_o + (size_t)pr * D + lane * PER;
#pragma unroll
    for (int i = 0; i < PER; ++i) acc[i] += wgt * src[i];
  }
  float denom = wsum;
  if (P.has_sinks) denom += ex2(P.sinks[head] * 1.4426950408889634f - Ms);
  const float inv = denom > 0.f ? 1.f / denom : 0.f;
  const int q_base = half ? P.d_q_indptr[req] : P.p_q_indptr[req];
  const size_t orow = (size_t)(q_base + tok) * P.H + head;
  T* out = reinterpret_cast<T*>(half ? P.out_d : P.out_p) + orow * D + lane * PER;
#pragma unroll
  for (int i = 0; i < PER; i += 2) {
    const uint32_t v = Pack<T>::two(acc[i] * inv, acc[i + 1] * inv);
    *reinterpret_cast<uint32_t*>(out + i) = v;
  }
  float* lse = half ? P.lse_d : P.lse_p;
  if (lane == 0 && lse) lse[orow] = wsum > 0.f ? M + log2f(wsum) : -INFINITY;
}

template <typename T, int D>
cudaError_t launch_merge(const PodParams& P, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  const int rows = P.counts_in_ws ? P.mrows_grid : P.n_mrows;
  cfg.gridDim = dim3((unsigned)((rows + 7) / 8));
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, pod_merge_kernel<T, D>, P);
}

}  // namespace

cudaError_t pod_launch(const PodParams& P, int dtype, cudaStream_t stream) {
  if (P.grid > 0) {
    // the host refuses a logits transform with an FP8 decode cache, and ALiBi
    // with RoPE; under RoPE a soft cap is a run-time switch of its kernel
    cudaError_t e = P.rope                  ? pod_k1_rope(P, dtype, stream)
                    : P.lt != POD_LT_NONE   ? pod_k1_lt(P, dtype, stream)
                                            : pod_k1_plain(P, dtype, stream);
    if (e != cudaSuccess) return e;
  }
  if ((P.counts_in_ws ? P.mrows_grid : P.n_mrows) > 0) {
    cudaError_t e;
    if (P.d == 256)
      e = dtype == 1 ? launch_merge<__nv_bfloat16, 256>(P, stream) : launch_merge<__half, 256>(P, stream);
    else if (P.d == 128)
      e = dtype == 1 ? launch_merge<__nv_bfloat16, 128>(P, stream) : launch_merge<__half, 128>(P, stream);
    else
      e = dtype == 1 ? launch_merge<__nv_bfloat16, 64>(P, stream) : launch_merge<__half, 64>(P, stream);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

int pod_kernel_smem_bytes(int d, int rope) { return rope ? pod_k1_smem_rope(d) : pod_k1_smem_plain(d); }
