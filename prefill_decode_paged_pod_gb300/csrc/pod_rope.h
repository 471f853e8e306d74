// pod_rope.h — host entry into the rotary-encoding pre-pass of pod_rope.cu.
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

// Angle per position of each pair j < d/2: (1 / rope_scale) * rope_theta^(-2j/d).
struct PodRopeFreq {
  double freq[128];
};

// The prefill half's cache: for every page-table entry, rotated K as a 16-bit
// high part and low part, and V copied, written compact (entry i -> page i
// of kv_dst, NHD [entries, 3, ps, Hk, d] with rows K_hi, V, K_lo).
struct PodRopeKV {
  const void* kv_src;          // the caller's cache, NHD or HND (hnd = 1)
  void* kv_dst;
  const int32_t* src_pages;    // [entries] the page-table entries
  const int32_t* ent;          // [entries][2] position of slot 0, slots below kv_len
  const float2* table;         // [rows][d/2] (cos, sin)
  int entries, ps, Hk, d, hnd;
};

// One half's queries: rotated copies of [rows, H, d] as high and low parts.
struct PodRopeQ {
  const void* q_src;
  void* q_hi;
  void* q_lo;
  const int32_t* qpos;         // [rows] position of each query row
  const float2* table;
  int rows, H, d;
};

cudaError_t pod_rope_table(float2* table, int rows, int half, const PodRopeFreq& f,
                           cudaStream_t stream);
cudaError_t pod_rope_kv(const PodRopeKV& a, int dtype, cudaStream_t stream);
cudaError_t pod_rope_q(const PodRopeQ& a, int dtype, cudaStream_t stream);
