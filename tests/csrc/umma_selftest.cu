// Self-test of the tcgen05 building blocks used by the POD prefill tile:
// 128B-swizzled shared-memory layouts written by cp.async, the shared-memory
// descriptors, the kind::f16 instruction descriptor, TMEM allocation and
// tcgen05.ld. One CTA computes
//   S = Q K^T   (M = 128, N = 64, K = D; both operands K-major)
//   O = P V     (M = 128, N = D, K = 64; V is MN-major)
// and writes S and O in fp32 so a test can compare them with torch matmuls.
// variant 0: O with one N = D MMA per k-step; variant 1: one N = 64 MMA per
// 64-column block of D; variant 2: P is written into TMEM (tcgen05.st, two
// 16-bit values per column) and read from there as the A operand.
// e4m3_selftest widens every pair of FP8 E4M3 codes with the decode path's
// conversion helper.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "pod_device.cuh"

using namespace pod;

template <int D, bool BF16>
__global__ void __launch_bounds__(128) umma_selftest_kernel(const uint16_t* q, const uint16_t* k,
                                                            const uint16_t* v, const uint16_t* p,
                                                            float* s_out, float* o_out,
                                                            int variant, int* status) {
  extern __shared__ __align__(1024) uint8_t smem[];
  constexpr int NKB = D / 64, QBLK = 128 * 128, KVBLK = 64 * 128;
  const uint32_t sb = smem_u32(smem);
  if ((sb & 1023u) != 0) {
    if (threadIdx.x == 0) *status = 2;
    return;
  }
  const uint32_t sQ = sb, sK = sQ + NKB * QBLK, sV = sK + NKB * KVBLK, sP = sV + NKB * KVBLK;
  const uint32_t bar = sP + 128 * 128;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + (bar - sb) + 64);
  const int tid = threadIdx.x, warp = tid >> 5;
  // operands -> swizzled shared memory
  for (int i = tid; i < 128 * (D / 8); i += 128) {
    int r = i / (D / 8), c = i % (D / 8);
    cp_async16(sQ + (c >> 3) * QBLK + sw128_off(r, c & 7), q + r * D + c * 8, 16);
  }
  for (int i = tid; i < 64 * (D / 8); i += 128) {
    int r = i / (D / 8), c = i % (D / 8);
    cp_async16(sK + (c >> 3) * KVBLK + sw128_off(r, c & 7), k + r * D + c * 8, 16);
    cp_async16(sV + (c >> 3) * KVBLK + sw128_off(r, c & 7), v + r * D + c * 8, 16);
  }
  for (int i = tid; i < 128 * 8; i += 128) {
    int r = i / 8, c = i % 8;
    cp_async16(sP + sw128_off(r, c), p + r * 64 + c * 8, 16);
  }
  cp_async_wait_all();
  fence_proxy_async();
  if (tid == 0) {
    mbar_init(bar, 1);
    mbar_init(bar + 8, 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(tslot), 256);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  if (variant == 2) {
    // row `tid` of P -> TMEM lane tid, columns 64..95 (S uses columns 0..63)
    uint32_t u[32];
    for (int i = 0; i < 32; ++i) u[i] = (uint32_t)p[tid * 64 + 2 * i] | ((uint32_t)p[tid * 64 + 2 * i + 1] << 16);
    tmem_st32u(tmem + ((uint32_t)(warp * 32) << 16) + 64, u);
    tmem_wait_st();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
  }
  if (tid == 0) {
    const uint32_t id_qk = idesc_f16(BF16, 128, 64, false, false);
    for (int kk = 0; kk < D / 16; ++kk) {
      uint64_t ad = sdesc_sw128(sQ + (kk >> 2) * QBLK + (kk & 3) * 32, 16, 1024);
      uint64_t bd = sdesc_sw128(sK + (kk >> 2) * KVBLK + (kk & 3) * 32, 16, 1024);
      mma_f16_ss(tmem + 0, ad, bd, id_qk, kk > 0);
    }
    mma_commit(bar);
    if (variant == 2) {
      const uint32_t id_pv = idesc_f16(BF16, 128, D, false, true);
      for (int kk = 0; kk < 4; ++kk) {
        uint64_t bd = sdesc_sw128(sV + kk * 2048, KVBLK, 1024);
        mma_f16_ts(tmem + 128, tmem + 64 + kk * 8, bd, id_pv, kk > 0);
      }
    } else if (variant == 0) {
      const uint32_t id_pv = idesc_f16(BF16, 128, D, false, true);
      for (int kk = 0; kk < 4; ++kk) {
        uint64_t ad = sdesc_sw128(sP + kk * 32, 16, 1024);
        uint64_t bd = sdesc_sw128(sV + kk * 2048, KVBLK, 1024);
        mma_f16_ss(tmem + 128, ad, bd, id_pv, kk > 0);
      }
    } else {
      const uint32_t id_pv = idesc_f16(BF16, 128, 64, false, true);
      for (int db = 0; db < NKB; ++db)
        for (int kk = 0; kk < 4; ++kk) {
          uint64_t ad = sdesc_sw128(sP + kk * 32, 16, 1024);
          uint64_t bd = sdesc_sw128(sV + db * KVBLK + kk * 2048, KVBLK, 1024);
          mma_f16_ss(tmem + 128 + db * 64, ad, bd, id_pv, kk > 0);
        }
    }
    mma_commit(bar + 8);
  }
  __syncwarp();
  volatile int never = 0;
  bool ok = mbar_wait(bar, 0, &never) && mbar_wait(bar + 8, 0, &never);
  tc_fence_after();
  const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
  const int row = tid;
  float buf[32];
  for (int c = 0; c < 64; c += 32) {
    tmem_ld32(tmem + lane_base + c, buf);
    for (int i = 0; i < 32; ++i) s_out[row * 64 + c + i] = buf[i];
  }
  for (int c = 0; c < D; c += 32) {
    tmem_ld32(tmem + lane_base + 128 + c, buf);
    for (int i = 0; i < 32; ++i) o_out[row * D + c + i] = buf[i];
  }
  if (!ok) atomicOr(status, 1);
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 256);
}

extern "C" int umma_selftest(const void* q, const void* k, const void* v, const void* p,
                             float* s_out, float* o_out, int d, int bf16, int variant,
                             int* status) {
  const int smem = (d / 64) * (128 * 128 + 2 * 64 * 128) + 128 * 128 + 256;
  auto launch = [&](auto kern) {
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    kern<<<1, 128, smem>>>((const uint16_t*)q, (const uint16_t*)k, (const uint16_t*)v,
                           (const uint16_t*)p, s_out, o_out, variant, status);
  };
  if (d == 128) {
    if (bf16) launch(umma_selftest_kernel<128, true>);
    else launch(umma_selftest_kernel<128, false>);
  } else {
    if (bf16) launch(umma_selftest_kernel<64, true>);
    else launch(umma_selftest_kernel<64, false>);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return (int)e;
  return (int)cudaDeviceSynchronize();
}

__global__ void e4m3_selftest_kernel(const uint16_t* in, uint32_t* out_h, uint32_t* out_b, int n) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) {
    out_h[i] = e4m3x2_to<__half>(in[i]);
    out_b[i] = e4m3x2_to<__nv_bfloat16>(in[i]);
  }
}

// n pairs of E4M3 codes (low byte first) -> packed fp16 pairs and bf16 pairs
extern "C" int e4m3_selftest(const void* in, void* out_h, void* out_b, int n) {
  e4m3_selftest_kernel<<<(n + 255) / 256, 256>>>((const uint16_t*)in, (uint32_t*)out_h,
                                                (uint32_t*)out_b, n);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return (int)e;
  return (int)cudaDeviceSynchronize();
}
