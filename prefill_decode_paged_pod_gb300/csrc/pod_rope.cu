// pod_rope.cu — rotary position encoding (ROPE_LLAMA): the pre-pass.
//
// Queries and keys are rotated at their positions before the dot product:
// query row i of a request at p = kv_len - q_len + i, key t at t; values are
// not rotated. Element j pairs with element j + d/2 and the pair turns by the
// angle (pos / rope_scale) * rope_theta^(-2j/d) (FlashInfer guide, "快速上手":
// pos_encoding_mode ROPE_LLAMA with rope_scale and rope_theta).
//
// A rotated value is not a 16-bit number. To keep the dot product as exact
// as the unrotated one, every rotated operand is stored as a 16-bit high
// part (the value rounded) and a 16-bit low part (the remainder rounded), and
// the kernels form q.k as q_hi.k_hi + q_hi.k_lo + q_lo.k_hi.
//
// These kernels write the rotated queries of both halves and, for the prefill
// half, copies of every page-table entry's page (K_hi, V, K_lo, NHD, in
// page-table order; the prefill page table for the kernels is the identity on
// them). Decode keys are rotated inside the fused kernel, straight from the
// caller's cache. The cos/sin table is computed once per bound workspace, in
// double precision, so long positions keep their accuracy.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "pod_rope.h"

namespace {

template <typename T>
struct Cvt;
template <>
struct Cvt<__half> {
  static __device__ float in(__half x) { return __half2float(x); }
  static __device__ __half out(float x) { return __float2half_rn(x); }
};
template <>
struct Cvt<__nv_bfloat16> {
  static __device__ float in(__nv_bfloat16 x) { return __bfloat162float(x); }
  static __device__ __nv_bfloat16 out(float x) { return __float2bfloat16_rn(x); }
};

// table[pos * half + j] = (cos, sin) of pos * freq[j]
__global__ void rope_table_kernel(float2* table, int rows, int half, PodRopeFreq f) {
  const long long n = (long long)rows * half;
  for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < n;
       idx += (long long)gridDim.x * blockDim.x) {
    const int j = (int)(idx % half);
    const long long pos = idx / half;
    double s, c;
    sincos((double)pos * f.freq[j], &s, &c);
    table[idx] = make_float2((float)c, (float)s);
  }
}

// Rotates 8 pairs (j0..j0+7 with j0+half..j0+half+7) of one row in fp32 and
// stores each result as a high part (dst_hi) and a low part (dst_lo).
template <typename T>
__device__ void rotate8(const T* src, T* dst_hi, T* dst_lo, int j0, int half, const float2* trow,
                        float sgn) {
  const uint4 a = *reinterpret_cast<const uint4*>(src + j0);
  const uint4 b = *reinterpret_cast<const uint4*>(src + j0 + half);
  const T* xa = reinterpret_cast<const T*>(&a);
  const T* xb = reinterpret_cast<const T*>(&b);
  uint4 ha, hb, la, lb;
  T* yha = reinterpret_cast<T*>(&ha);
  T* yhb = reinterpret_cast<T*>(&hb);
  T* yla = reinterpret_cast<T*>(&la);
  T* ylb = reinterpret_cast<T*>(&lb);
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    const float2 cs = trow[j0 + e];
    const float c = cs.x, sn = sgn * cs.y;
    const float u = Cvt<T>::in(xa[e]), v = Cvt<T>::in(xb[e]);
    const float ru = fmaf(u, c, -v * sn), rv = fmaf(v, c, u * sn);
    yha[e] = Cvt<T>::out(ru);
    yhb[e] = Cvt<T>::out(rv);
    yla[e] = Cvt<T>::out(ru - Cvt<T>::in(yha[e]));
    ylb[e] = Cvt<T>::out(rv - Cvt<T>::in(yhb[e]));
  }
  *reinterpret_cast<uint4*>(dst_hi + j0) = ha;
  *reinterpret_cast<uint4*>(dst_hi + j0 + half) = hb;
  *reinterpret_cast<uint4*>(dst_lo + j0) = la;
  *reinterpret_cast<uint4*>(dst_lo + j0 + half) = lb;
}

// One thread per (page-table entry, slot, kv head, 8-pair chunk): rotates the
// K row into its high and low rows, copies the V row, into the compact NHD
// copy [entries, 3, ps, Hk, d] (rows K_hi, V, K_lo). Slots at or past the
// request's kv_len are written as zeros.
template <typename T>
__global__ void rope_kv_kernel(PodRopeKV a) {
  const int half = a.d / 2, chunks = half / 8;
  const long long n = (long long)a.entries * a.ps * a.Hk * chunks;
  const T* src = static_cast<const T*>(a.kv_src);
  T* dst = static_cast<T*>(a.kv_dst);
  const long long rowstride = (long long)a.ps * a.Hk * a.d;   // K -> V -> K_lo rows
  for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < n;
       idx += (long long)gridDim.x * blockDim.x) {
    const int cj = (int)(idx % chunks);
    long long r = idx / chunks;
    const int hk = (int)(r % a.Hk);
    r /= a.Hk;
    const int s = (int)(r % a.ps);
    const int i = (int)(r / a.ps);
    const long long page = a.src_pages[i];
    const int pos0 = a.ent[2 * i], valid = a.ent[2 * i + 1];
    const long long ks = a.hnd ? (((page * 2 + 0) * a.Hk + hk) * a.ps + s) * a.d
                               : (((page * 2 + 0) * a.ps + s) * a.Hk + hk) * a.d;
    const long long vs = ks + rowstride;                      // the V half of the source page
    const long long kd = ((long long)i * 3 * a.ps + s) * a.Hk * a.d + (long long)hk * a.d;
    const long long vd = kd + rowstride, ld = kd + 2 * rowstride;
    const int j0 = cj * 8;
    if (s < valid) {
      rotate8<T>(src + ks, dst + kd, dst + ld, j0, half, a.table + (long long)(pos0 + s) * half, 1.f);
      *reinterpret_cast<uint4*>(dst + vd + j0) = *reinterpret_cast<const uint4*>(src + vs + j0);
      *reinterpret_cast<uint4*>(dst + vd + j0 + half) =
          *reinterpret_cast<const uint4*>(src + vs + j0 + half);
    } else {
      const uint4 z = make_uint4(0u, 0u, 0u, 0u);
      const long long rows3[3] = {kd, vd, ld};
      for (int q = 0; q < 3; ++q) {
        *reinterpret_cast<uint4*>(dst + rows3[q] + j0) = z;
        *reinterpret_cast<uint4*>(dst + rows3[q] + j0 + half) = z;
      }
    }
  }
}

// One thread per (query row, qo head, 8-pair chunk); a negative position
// turns the other way (cos is even, sin odd).
template <typename T>
__global__ void rope_q_kernel(PodRopeQ a) {
  const int half = a.d / 2, chunks = half / 8;
  const long long n = (long long)a.rows * a.H * chunks;
  const T* src = static_cast<const T*>(a.q_src);
  T* hi = static_cast<T*>(a.q_hi);
  T* lo = static_cast<T*>(a.q_lo);
  for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < n;
       idx += (long long)gridDim.x * blockDim.x) {
    const int cj = (int)(idx % chunks);
    const long long rh = idx / chunks;               // row * H + head
    const int pos = a.qpos[rh / a.H];
    const int apos = pos < 0 ? -pos : pos;
    rotate8<T>(src + rh * a.d, hi + rh * a.d, lo + rh * a.d, cj * 8, half,
               a.table + (long long)apos * half, pos < 0 ? -1.f : 1.f);
  }
}

int blocks_for(long long n) {
  long long b = (n + 255) / 256;
  return (int)(b < 1 ? 1 : (b > 152 * 32 ? 152 * 32 : b));
}

}  // namespace

cudaError_t pod_rope_table(float2* table, int rows, int half, const PodRopeFreq& f,
                           cudaStream_t stream) {
  rope_table_kernel<<<blocks_for((long long)rows * half), 256, 0, stream>>>(table, rows, half, f);
  return cudaGetLastError();
}

cudaError_t pod_rope_kv(const PodRopeKV& a, int dtype, cudaStream_t stream) {
  const long long n = (long long)a.entries * a.ps * a.Hk * (a.d / 16);
  if (n == 0) return cudaSuccess;
  if (dtype == 1)
    rope_kv_kernel<__nv_bfloat16><<<blocks_for(n), 256, 0, stream>>>(a);
  else
    rope_kv_kernel<__half><<<blocks_for(n), 256, 0, stream>>>(a);
  return cudaGetLastError();
}

cudaError_t pod_rope_q(const PodRopeQ& a, int dtype, cudaStream_t stream) {
  const long long n = (long long)a.rows * a.H * (a.d / 16);
  if (n == 0) return cudaSuccess;
  if (dtype == 1)
    rope_q_kernel<__nv_bfloat16><<<blocks_for(n), 256, 0, stream>>>(a);
  else
    rope_q_kernel<__half><<<blocks_for(n), 256, 0, stream>>>(a);
  return cudaGetLastError();
}
