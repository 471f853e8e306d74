// pod_api.cu — the extern "C" boundary declared in include/pod.h.
//
// Host-side only: argument checks, the planner call, the one metadata upload
// and the kernel launches. Every step of the attention itself runs in the
// kernels (pod_kernels.cuh, launched through pod_launch.cu).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <algorithm>
#include <cmath>
#include <new>
#include <string>

#include "../../include/pod.h"
#include "pod_launch.h"
#include "pod_planner.hpp"
#include "pod_rope.h"

struct pod_plan_s {
  PodPlanHost plan;
  // decode cache stored as FP8 E4M3 codes with per-tensor K and V scales
  int d_fp8 = 0;
  float k_scale = 1.f, v_scale = 1.f;
  // page layout of each half's cache: 0 = NHD, 1 = HND
  int p_layout = 0, d_layout = 0;
  // logits transform of both halves: soft cap (> 0) or ALiBi slopes (device [H])
  float soft_cap = 0.f;
  const float* alibi = nullptr;
  // custom prefill mask: caller-owned device bytes read by every run
  const void* p_mask = nullptr;
  int64_t p_mask_bytes = 0;
  // RoPE: the workspace whose cos/sin table is filled (nullptr: none yet)
  const void* rope_table_ws = nullptr;
  void* workspace = nullptr;      // bound device workspace (nullptr = host-only plan)
  size_t workspace_bytes = 0;
  // TMA descriptors of the last run, re-encoded only when a tensor pointer
  // changes: q_p, kv_p, q_d, kv_d, then (RoPE) the low parts of q_p and q_d
  const void* tm_ptr[6] = {nullptr, nullptr, nullptr, nullptr, nullptr, nullptr};
  CUtensorMap tm[6];
};

namespace {

thread_local std::string g_err;

pod_status set_err(pod_status code, const std::string& msg) {
  g_err = msg;
  return code;
}

pod_status cuda_err(cudaError_t e, const char* what) {
  return set_err(POD_ERR_CUDA, std::string(what) + ": " + cudaGetErrorString(e));
}

int log_level() {
  static int lvl = -1;
  if (lvl < 0) {
    const char* s = getenv("POD_LOGLEVEL");
    lvl = s ? atoi(s) : 0;
  }
  return lvl;
}

pod_status upload(pod_plan_s* h, void* ws, size_t bytes, void* stream) {
  const PodPlanHost& P = h->plan;
  if (ws == nullptr || bytes < P.total_bytes)
    return set_err(POD_ERR_WORKSPACE, "workspace of " + std::to_string(bytes) +
                                          " bytes is smaller than the plan's " +
                                          std::to_string(P.total_bytes));
  if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0)
    return set_err(POD_ERR_WORKSPACE, "workspace must be 256-byte aligned");
  cudaError_t e = cudaMemcpyAsync(ws, P.int_image.data(), P.int_image.size(),
                                  cudaMemcpyHostToDevice, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_err(e, "cudaMemcpyAsync(plan metadata)");
  // the copy reads pageable host memory owned by the handle: finish it before returning
  e = cudaStreamSynchronize((cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_err(e, "cudaStreamSynchronize(plan metadata)");
  h->workspace = ws;
  h->workspace_bytes = bytes;
  h->rope_table_ws = nullptr;
  return POD_OK;
}

// ---- TMA descriptors (driver entry point fetched through the runtime) --------
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// Q viewed as [rows][H][d]; box = 64 elements x G heads x `tokens` rows.
pod_status encode_q(CUtensorMap* m, const void* ptr, int rows, int H, int d, int G, int tokens,
                    int dtype) {
  auto fn = encode_fn();
  if (!fn) return set_err(POD_ERR_CUDA, "cuTensorMapEncodeTiled is not available");
  if ((reinterpret_cast<uintptr_t>(ptr) & 15u) != 0)
    return set_err(POD_ERR_INVALID_ARG, "q tensors must be 16-byte aligned");
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)H, (cuuint64_t)rows};
  cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)H * d * 2};
  cuuint32_t box[3] = {64, (cuuint32_t)G, (cuuint32_t)tokens};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(m, dtype ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
                  const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return set_err(POD_ERR_CUDA, "cuTensorMapEncodeTiled(q) failed: " + std::to_string((int)r));
  return POD_OK;
}

// Paged cache viewed as [pages][nkv][ps][Hk][d] (dims listed the same way for
// an HND cache, [pages][nkv][Hk][ps][d] in memory, with its strides); nkv = 2
// (K, V), or 3 for the RoPE prefill copies (K_hi, V, K_lo). A box holds `kbx`
// keys: 64 elements x 1 head x kbx slots x 1 x 1 page when ps >= 8
// (kbx <= ps), or 64 x 1 x ps slots x 1 x (kbx / ps) pages when ps < 8.
pod_status encode_kv(CUtensorMap* m, const void* ptr, int num_pages, int ps, int Hk, int d,
                     int kbx, int dtype, int hnd, int nkv) {
  auto fn = encode_fn();
  if (!fn) return set_err(POD_ERR_CUDA, "cuTensorMapEncodeTiled is not available");
  if ((reinterpret_cast<uintptr_t>(ptr) & 15u) != 0)
    return set_err(POD_ERR_INVALID_ARG, "kv caches must be 16-byte aligned");
  cuuint64_t dims[5] = {(cuuint64_t)d, (cuuint64_t)Hk, (cuuint64_t)ps, (cuuint64_t)nkv,
                        (cuuint64_t)num_pages};
  cuuint64_t row = (cuuint64_t)d * 2;
  // the same logical dims for both layouts; HND swaps the head and slot strides
  cuuint64_t strides[4] = {hnd ? row * ps : row, hnd ? row : row * Hk, row * Hk * ps,
                           row * Hk * ps * nkv};
  cuuint32_t box[5] = {64, 1, (cuuint32_t)(ps >= 8 ? kbx : ps), 1,
                       (cuuint32_t)(ps >= 8 ? 1 : kbx / ps)};
  cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  CUresult r = fn(m, dtype ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 5,
                  const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return set_err(POD_ERR_CUDA, "cuTensorMapEncodeTiled(kv) failed: " + std::to_string((int)r));
  return POD_OK;
}

// Decode view of the paged cache: one box holds `kbx` keys of one head with
// both 64-element halves of head_dim, landing in shared memory as
// [half][key][64] (each half a run of kbx 128-byte rows). Dims, innermost
// first: page_size >= 8: [64][ps][d/64][Hk][2 * pages] (K/V and page merged:
// coordinate 2 * page + kv); page_size 1: [64][pages][d/64][Hk][2] (an HND
// cache has the same bytes there). HND swaps the slot and head strides.
pod_status encode_kv_decode(CUtensorMap* m, const void* ptr, int num_pages, int ps, int Hk, int d,
                            int kbx, int dtype, int hnd) {
  auto fn = encode_fn();
  if (!fn) return set_err(POD_ERR_CUDA, "cuTensorMapEncodeTiled is not available");
  if ((reinterpret_cast<uintptr_t>(ptr) & 15u) != 0)
    return set_err(POD_ERR_INVALID_ARG, "kv caches must be 16-byte aligned");
  const cuuint64_t row = (cuuint64_t)d * 2, nh = (cuuint64_t)d / 64;
  cuuint64_t dims[5], strides[4];
  if (ps >= 8) {
    cuuint64_t d5[5] = {64, (cuuint64_t)ps, nh, (cuuint64_t)Hk, 2 * (cuuint64_t)num_pages};
    cuuint64_t s4[4] = {hnd ? row : row * Hk, 128, hnd ? row * ps : row, row * Hk * ps};
    memcpy(dims, d5, sizeof(d5));
    memcpy(strides, s4, sizeof(s4));
  } else {
    cuuint64_t d5[5] = {64, (cuuint64_t)num_pages, nh, (cuuint64_t)Hk, 2};
    cuuint64_t s4[4] = {row * Hk * 2, 128, row, row * Hk};
    memcpy(dims, d5, sizeof(d5));
    memcpy(strides, s4, sizeof(s4));
  }
  cuuint32_t box[5] = {64, (cuuint32_t)kbx, (cuuint32_t)nh, 1, 1};
  cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  CUresult r = fn(m, dtype ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 5,
                  const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return set_err(POD_ERR_CUDA, "cuTensorMapEncodeTiled(kv, decode) failed: " + std::to_string((int)r));
  return POD_OK;
}

// FP8 (E4M3) decode view of the paged cache: a key's head row is 128 bytes,
// one 128-byte swizzle row; one box holds `kbx` keys of one head and lands as
// [key][128]. Dims, innermost first: page_size >= 8:
// [128][ps][Hk][2 * pages] (coordinate 2 * page + kv); page_size 1:
// [128][pages][Hk][2].
pod_status encode_kv_decode_fp8(CUtensorMap* m, const void* ptr, int num_pages, int ps, int Hk,
                                int d, int kbx, int hnd) {
  auto fn = encode_fn();
  if (!fn) return set_err(POD_ERR_CUDA, "cuTensorMapEncodeTiled is not available");
  if ((reinterpret_cast<uintptr_t>(ptr) & 15u) != 0)
    return set_err(POD_ERR_INVALID_ARG, "kv caches must be 16-byte aligned");
  const cuuint64_t row = (cuuint64_t)d;  // bytes per head row
  cuuint64_t dims[4], strides[3];
  if (ps >= 8) {
    cuuint64_t d4[4] = {(cuuint64_t)d, (cuuint64_t)ps, (cuuint64_t)Hk, 2 * (cuuint64_t)num_pages};
    cuuint64_t s3[3] = {hnd ? row : row * Hk, hnd ? row * ps : row, row * Hk * ps};
    memcpy(dims, d4, sizeof(d4));
    memcpy(strides, s3, sizeof(s3));
  } else {
    cuuint64_t d4[4] = {(cuuint64_t)d, (cuuint64_t)num_pages, (cuuint64_t)Hk, 2};
    cuuint64_t s3[3] = {row * Hk * 2, row, row * Hk};
    memcpy(dims, d4, sizeof(d4));
    memcpy(strides, s3, sizeof(s3));
  }
  cuuint32_t box[4] = {(cuuint32_t)d, (cuuint32_t)kbx, 1, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(ptr), dims, strides, box,
                  estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return set_err(POD_ERR_CUDA, "cuTensorMapEncodeTiled(kv, decode fp8) failed: " + std::to_string((int)r));
  return POD_OK;
}

// Plan arguments that rebuild `O` from the handle's own copies of the page
// tables (the optional switches can then be changed one at a time).
PodPlanArgs args_of(const PodPlanHost& O) {
  PodPlanArgs a;
  a.p_q_indptr = O.p.q_indptr.data(); a.p_kv_indptr = O.p.kv_indptr.data();
  a.p_kv_indices = O.p.kv_indices.data(); a.p_last_page_len = O.p.last_page_len.data();
  a.p_batch = O.p.batch; a.p_num_pages = O.p.num_pages;
  a.d_q_indptr = O.dd.q_indptr.data(); a.d_kv_indptr = O.dd.kv_indptr.data();
  a.d_kv_indices = O.dd.kv_indices.data(); a.d_last_page_len = O.dd.last_page_len.data();
  a.d_batch = O.dd.batch; a.d_num_pages = O.dd.num_pages;
  a.H = O.H; a.Hk = O.Hk; a.d = O.d; a.ps = O.ps; a.causal = O.causal;
  a.window_left = O.window_left; a.sm_scale = O.sm_scale; a.dtype = O.dtype;
  a.has_sinks = O.has_sinks; a.num_sms = O.num_sms; a.p_custom_mask = O.p_custom_mask;
  a.rope = O.rope; a.rope_scale = O.rope_scale; a.rope_theta = O.rope_theta;
  a.graph = O.graph;
  a.cap_p_batch = O.cap_p_batch; a.cap_p_rows = O.cap_p_rows; a.cap_p_pages = O.cap_p_pages;
  a.cap_d_batch = O.cap_d_batch; a.cap_d_rows = O.cap_d_rows; a.cap_d_pages = O.cap_d_pages;
  return a;
}

// Replaces the handle's plan by one made from `a`; the layout may change, so
// any bound workspace is released (the caller binds again).
pod_status replan(pod_plan_s* h, const PodPlanArgs& a) {
  PodPlanHost fresh;
  std::string err;
  const int rc = pod_build_plan(a, fresh, &err);
  if (rc != 0) return set_err((pod_status)rc, err);
  h->plan = std::move(fresh);
  h->workspace = nullptr;
  h->workspace_bytes = 0;
  h->rope_table_ws = nullptr;
  for (int i = 0; i < 6; ++i) h->tm_ptr[i] = nullptr;
  return POD_OK;
}

}  // namespace

// Lets other translation units of the library report a message through
// pod_last_error().
void pod_set_last_error(const std::string& msg) { g_err = msg; }

extern "C" {

pod_status pod_plan(const int32_t* p_q_indptr, const int32_t* p_kv_indptr,
                    const int32_t* p_kv_indices, const int32_t* p_last_page_len, int32_t p_batch,
                    int32_t p_num_pages, const int32_t* d_q_indptr, const int32_t* d_kv_indptr,
                    const int32_t* d_kv_indices, const int32_t* d_last_page_len, int32_t d_batch,
                    int32_t d_num_pages, int32_t num_qo_heads, int32_t num_kv_heads,
                    int32_t head_dim, int32_t page_size, int32_t causal, int32_t window_left,
                    float sm_scale, pod_dtype dtype, int32_t has_sinks, int32_t num_sms,
                    void* workspace, size_t workspace_bytes, void* stream,
                    pod_handle* out_handle, size_t* required_workspace_bytes) {
  g_err.clear();
  if (!out_handle) return set_err(POD_ERR_INVALID_ARG, "out_handle is NULL");
  *out_handle = nullptr;
  if (required_workspace_bytes) *required_workspace_bytes = 0;
  if (num_sms <= 0) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_err(e, "cudaGetDevice");
    e = cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_err(e, "cudaDeviceGetAttribute(SM count)");
  }
  PodPlanArgs a;
  a.p_q_indptr = p_q_indptr; a.p_kv_indptr = p_kv_indptr; a.p_kv_indices = p_kv_indices;
  a.p_last_page_len = p_last_page_len; a.p_batch = p_batch; a.p_num_pages = p_num_pages;
  a.d_q_indptr = d_q_indptr; a.d_kv_indptr = d_kv_indptr; a.d_kv_indices = d_kv_indices;
  a.d_last_page_len = d_last_page_len; a.d_batch = d_batch; a.d_num_pages = d_num_pages;
  a.H = num_qo_heads; a.Hk = num_kv_heads; a.d = head_dim; a.ps = page_size;
  a.causal = causal; a.window_left = window_left; a.sm_scale = sm_scale;
  a.dtype = (int)dtype; a.has_sinks = has_sinks; a.num_sms = num_sms;
  a.p_custom_mask = 0;
  a.rope = 0; a.rope_scale = 1.0; a.rope_theta = 1e4;
  a.graph = 0;
  a.cap_p_batch = a.cap_p_rows = a.cap_p_pages = a.cap_d_batch = a.cap_d_rows = a.cap_d_pages = 0;

  pod_plan_s* h = new (std::nothrow) pod_plan_s();
  if (!h) return set_err(POD_ERR_INVALID_ARG, "out of host memory");
  std::string err;
  int rc = pod_build_plan(a, h->plan, &err);
  if (rc != 0) {
    delete h;
    return set_err((pod_status)rc, err);
  }
  if (required_workspace_bytes) *required_workspace_bytes = h->plan.total_bytes;
  if (workspace != nullptr) {
    pod_status st = upload(h, workspace, workspace_bytes, stream);
    if (st != POD_OK) {
      delete h;
      return st;
    }
  }
  if (log_level() >= 1) {
    const PodPlanHost& P = h->plan;
    fprintf(stderr,
            "[pod] plan: H=%d Hk=%d d=%d ps=%d causal=%d window=%d | prefill rows=%d tiles=%zu "
            "ctas=%d | decode rows=%d items=%zu ctas=%d chunk=%d | merge rows=%d | workspace=%zu B\n",
            P.H, P.Hk, P.d, P.ps, P.causal, P.window_left, P.p.rows, P.ptiles.size() / POD_REC,
            P.n_p_ctas, P.dd.rows, P.ditems.size() / POD_REC, P.n_d_ctas, P.decode_chunk,
            P.n_mrows, P.total_bytes);
  }
  *out_handle = h;
  return POD_OK;
}

size_t pod_workspace_size(pod_handle h) { return h ? h->plan.total_bytes : 0; }

pod_status pod_bind_workspace(pod_handle h, void* workspace, size_t workspace_bytes, void* stream) {
  g_err.clear();
  if (!h) return set_err(POD_ERR_INVALID_ARG, "handle is NULL");
  return upload(h, workspace, workspace_bytes, stream);
}

pod_status pod_run(pod_handle h, const void* q_p, const void* kv_p, const void* q_d,
                   const void* kv_d, const float* sinks, void* workspace, void* out_p,
                   float* lse_p, void* out_d, float* lse_d, void* stream) {
  g_err.clear();
  if (!h) return set_err(POD_ERR_INVALID_ARG, "handle is NULL");
  const PodPlanHost& P = h->plan;
  if (!h->workspace) return set_err(POD_ERR_WORKSPACE, "the plan has no bound workspace");
  if (workspace != h->workspace)
    return set_err(POD_ERR_WORKSPACE, "workspace differs from the one the plan was bound to");
  // capacity mode: a captured launch replays later plans, so every half with
  // a capacity needs its tensors (sized for the capacity) on every run
  const int p_rows_t = P.graph ? P.cap_p_rows : P.p.rows;
  const int d_rows_t = P.graph ? P.cap_d_rows : P.dd.rows;
  if (p_rows_t > 0 && (!q_p || !kv_p || !out_p))
    return set_err(POD_ERR_INVALID_ARG, "prefill half is non-empty but q_p/kv_p/out_p is NULL");
  if (d_rows_t > 0 && (!q_d || !kv_d || !out_d))
    return set_err(POD_ERR_INVALID_ARG, "decode half is non-empty but q_d/kv_d/out_d is NULL");
  if (P.has_sinks && !sinks) return set_err(POD_ERR_INVALID_ARG, "plan has sinks but sinks is NULL");
  if (!P.has_sinks && sinks)
    return set_err(POD_ERR_INVALID_ARG, "sinks given but the plan was made without sinks");
  if (h->alibi) {
    cudaPointerAttributes pa;
    cudaError_t e = cudaPointerGetAttributes(&pa, h->alibi);
    if (e != cudaSuccess) return cuda_err(e, "cudaPointerGetAttributes(alibi slopes)");
    if (pa.type != cudaMemoryTypeDevice && pa.type != cudaMemoryTypeManaged)
      return set_err(POD_ERR_INVALID_ARG, "the ALiBi slopes are not device memory");
  }
  if (P.p_custom_mask && P.p.rows > 0) {
    // the kernel reads the mask: it must be device (or managed) memory
    cudaPointerAttributes pa;
    cudaError_t e = cudaPointerGetAttributes(&pa, h->p_mask);
    if (e != cudaSuccess) return cuda_err(e, "cudaPointerGetAttributes(prefill mask)");
    if (pa.type != cudaMemoryTypeDevice && pa.type != cudaMemoryTypeManaged)
      return set_err(POD_ERR_INVALID_ARG, "the custom prefill mask is not device memory");
  }

  uint8_t* ws = static_cast<uint8_t*>(workspace);
  // RoPE: the rotated queries of both halves (high and low parts) and copies
  // of the prefill half's pages (K_hi, V, K_lo) are written into the
  // workspace; the kernels read those, and rotate the decode keys themselves
  int p_layout = h->p_layout, d_layout = h->d_layout;
  int p_pages = P.p.num_pages, d_pages = P.dd.num_pages;
  const void* q_p_lo = nullptr;
  const void* q_d_lo = nullptr;
  const float2* rope_tab = nullptr;
  if (P.rope) {
    cudaStream_t st = (cudaStream_t)stream;
    rope_tab = reinterpret_cast<const float2*>(ws + P.off_rope_table);
    if (h->rope_table_ws != workspace) {
      PodRopeFreq f;
      for (int j = 0; j < P.d / 2; ++j)
        f.freq[j] = std::pow(P.rope_theta, -2.0 * j / P.d) / P.rope_scale;
      cudaError_t e = pod_rope_table(reinterpret_cast<float2*>(ws + P.off_rope_table), P.rope_rows,
                                     P.d / 2, f, st);
      if (e != cudaSuccess) return cuda_err(e, "RoPE table launch");
      h->rope_table_ws = workspace;
    }
    const void* srcs[4] = {q_p, kv_p, q_d, kv_d};
    for (const void* p : srcs)
      if ((reinterpret_cast<uintptr_t>(p) & 15u) != 0)
        return set_err(POD_ERR_INVALID_ARG, "q and kv tensors must be 16-byte aligned");
    auto I32 = [&](size_t off) { return reinterpret_cast<const int32_t*>(ws + off); };
    for (int half = 0; half < 2; ++half) {
      const PodHalfHost& hh = half ? P.dd : P.p;
      if (hh.rows == 0) continue;
      PodRopeQ q;
      q.q_src = half ? q_d : q_p;
      q.q_hi = ws + (half ? P.off_d_qcopy : P.off_p_qcopy);
      q.q_lo = ws + (half ? P.off_d_qcopy_lo : P.off_p_qcopy_lo);
      q.qpos = I32(half ? P.off_d_rope_qpos : P.off_p_rope_qpos);
      q.table = rope_tab;
      q.rows = hh.rows; q.H = P.H; q.d = P.d;
      cudaError_t e = pod_rope_q(q, P.dtype, st);
      if (e != cudaSuccess) return cuda_err(e, "RoPE query launch");
    }
    if (P.p.rows > 0) {
      PodRopeKV k;
      k.kv_src = kv_p;
      k.kv_dst = ws + P.off_p_kvcopy;
      k.src_pages = I32(P.off_p_rope_src);
      k.ent = I32(P.off_p_rope_ent);
      k.table = rope_tab;
      k.entries = (int)P.p.kv_indices.size(); k.ps = P.ps; k.Hk = P.Hk; k.d = P.d;
      k.hnd = h->p_layout;
      cudaError_t e = pod_rope_kv(k, P.dtype, st);
      if (e != cudaSuccess) return cuda_err(e, "RoPE prefill key launch");
    }
    q_p = ws + P.off_p_qcopy; kv_p = ws + P.off_p_kvcopy;
    q_p_lo = ws + P.off_p_qcopy_lo;
    q_d = ws + P.off_d_qcopy;
    q_d_lo = ws + P.off_d_qcopy_lo;
    p_layout = 0;
    p_pages = (int)P.p.kv_indices.size();
  }

  // TMA descriptors for the tensors of this call (cached while pointers repeat)
  const void* ptrs[6] = {q_p, kv_p, q_d, kv_d, q_p_lo, q_d_lo};
  for (int i = 0; i < 6; ++i) {
    const bool pre = i < 2 || i == 4;
    const int rows = pre ? p_rows_t : d_rows_t;   // the q tensor's rows
    if (rows == 0) continue;
    if (i >= 4 && !P.rope) continue;
    if ((i == 1 || i == 3) && !(pre ? P.p_tma : P.d_tma)) continue;
    if (h->tm_ptr[i] == ptrs[i]) continue;
    const int npages = pre ? p_pages : d_pages;
    pod_status st;
    if (i == 0 || i == 2 || i >= 4)
      st = encode_q(&h->tm[i], ptrs[i], rows, P.H, P.d, P.G, pre ? P.tq : P.tu, P.dtype);
    else if (pre)
      st = encode_kv(&h->tm[i], ptrs[i], npages, P.ps, P.Hk, P.d, P.p_tma, P.dtype, p_layout,
                     P.rope ? 3 : 2);
    else if (h->d_fp8)
      st = encode_kv_decode_fp8(&h->tm[i], ptrs[i], npages, P.ps, P.Hk, P.d, P.d_tma, d_layout);
    else
      st = encode_kv_decode(&h->tm[i], ptrs[i], npages, P.ps, P.Hk, P.d, P.d_tma, P.dtype, d_layout);
    if (st != POD_OK) return st;
    h->tm_ptr[i] = ptrs[i];
  }

  PodParams K;
  memset(&K, 0, sizeof(K));
  if (p_rows_t) {
    K.tm_q_p = h->tm[0];
    if (P.p_tma) K.tm_kv_p = h->tm[1];
  }
  if (d_rows_t) {
    K.tm_q_d = h->tm[2];
    if (P.d_tma) K.tm_kv_d = h->tm[3];
  }
  if (P.rope) {
    if (P.p.rows) K.tm_qlo_p = h->tm[4];
    if (P.dd.rows) K.tm_qlo_d = h->tm[5];
    K.rope = 1;
    K.rope_rows = P.rope_rows;
    K.rope_tab = rope_tab;
    K.q_d_lo = q_d_lo;
  }
  K.p_tma = P.p_tma;
  K.d_tma = P.d_tma;
  K.p_num_pages = p_pages;
  K.d_num_pages = d_pages;
  K.tq = P.tq;
  K.tu = P.tu;
  K.H = P.H; K.Hk = P.Hk; K.G = P.G; K.d = P.d; K.ps = P.ps;
  K.ps_shift = -1;
  for (int s = 0; s < 31; ++s)
    if ((1 << s) == P.ps) K.ps_shift = s;
  K.causal = P.causal; K.window_left = P.window_left; K.has_sinks = P.has_sinks;
  K.p_hnd = p_layout;
  K.d_hnd = d_layout;
  K.lt = h->soft_cap > 0.f ? POD_LT_SOFTCAP : (h->alibi ? POD_LT_ALIBI : POD_LT_NONE);
  K.lt_c = h->soft_cap / P.sm_scale;
  K.lt_inv_scale = 1.f / P.sm_scale;
  K.alibi = h->alibi;
  K.scale_log2 = P.scale_log2;
  K.d_fp8 = h->d_fp8;
  K.d_scale_log2 = P.scale_log2 * h->k_scale;
  K.v_scale = h->v_scale;
  K.n_p_ctas = P.n_p_ctas; K.grid = P.grid;
  K.n_groups = (int)(P.mgroups.size() / POD_REC); K.n_mrows = P.n_mrows;
  // CUDA-graph capacity mode: counts from the workspace, merge grid for the
  // capacity's merge rows
  K.counts_in_ws = P.graph;
  K.mrows_grid = P.cap_mrows;
  K.p_batch = P.p.batch; K.d_batch = P.dd.batch;
  auto I = [&](size_t off) { return reinterpret_cast<const int32_t*>(ws + off); };
  K.p_q_indptr = I(P.off_p_q_indptr); K.p_kv_indptr = I(P.off_p_kv_indptr);
  K.p_kv_indices = I(P.off_p_kv_indices); K.p_kv_len = I(P.off_p_kv_len);
  K.d_q_indptr = I(P.off_d_q_indptr); K.d_kv_indptr = I(P.off_d_kv_indptr);
  K.d_kv_indices = I(P.off_d_kv_indices); K.d_kv_len = I(P.off_d_kv_len);
  K.ptiles = I(P.off_ptiles); K.ditems = I(P.off_ditems);
  K.cta_ptr = I(P.off_cta_ptr); K.cta_list = I(P.off_cta_list);
  K.mgroups = I(P.off_mgroups); K.mrow_ptr = I(P.off_mrow_ptr);
  K.pqueue = I(P.off_pqueue); K.dqueue = I(P.off_dqueue); K.dqrec = I(P.off_dqrec);
  // capacity mode: the queues' capacities (sentinels follow the plan's records)
  K.n_tiles = P.graph ? P.cap_tiles : (int)P.pqueue.size();
  K.n_items = P.graph ? P.cap_items : (int)P.dqueue.size();
  K.part_o = reinterpret_cast<float*>(ws + P.off_part_o);
  K.part_lse = reinterpret_cast<float*>(ws + P.off_part_lse);
  K.status = reinterpret_cast<int32_t*>(ws + P.off_status);
  K.q_p = q_p; K.kv_p = kv_p; K.q_d = q_d; K.kv_d = kv_d; K.sinks = sinks;
  if (P.p_custom_mask && P.p.rows > 0) {
    K.p_mask = static_cast<const uint8_t*>(h->p_mask);
    K.p_mask_off = reinterpret_cast<const long long*>(ws + P.off_p_mask_off);
    K.p_mask_bytes = (long long)h->p_mask_bytes;
  }
  K.out_p = out_p; K.out_d = out_d; K.lse_p = lse_p; K.lse_d = lse_d;

  cudaError_t e = pod_launch(K, P.dtype, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_err(e, "kernel launch");
  return POD_OK;
}

pod_status pod_destroy(pod_handle h) {
  delete h;
  return POD_OK;
}

pod_status pod_plan_set_decode_fp8(pod_handle h, float k_scale, float v_scale) {
  g_err.clear();
  if (!h) return set_err(POD_ERR_INVALID_ARG, "handle is NULL");
  if (h->plan.d != 128)
    return set_err(POD_ERR_UNSUPPORTED, "an FP8 decode cache needs head_dim 128");
  if (!(k_scale > 0.f) || !(v_scale > 0.f) || !std::isfinite(k_scale) || !std::isfinite(v_scale))
    return set_err(POD_ERR_INVALID_ARG, "k_scale and v_scale must be finite and positive");
  if (h->soft_cap > 0.f || h->alibi)
    return set_err(POD_ERR_UNSUPPORTED, "an FP8 decode cache with a soft cap or ALiBi");
  if (h->plan.rope) return set_err(POD_ERR_UNSUPPORTED, "an FP8 decode cache with RoPE");
  h->d_fp8 = 1;
  h->k_scale = k_scale;
  h->v_scale = v_scale;
  h->tm_ptr[3] = nullptr;  // the decode cache's tensor map changes format
  return POD_OK;
}

pod_status pod_plan_set_logits_transform(pod_handle h, float logits_soft_cap,
                                         const float* alibi_slopes) {
  g_err.clear();
  if (!h) return set_err(POD_ERR_INVALID_ARG, "handle is NULL");
  if (!std::isfinite(logits_soft_cap) || logits_soft_cap < 0.f)
    return set_err(POD_ERR_INVALID_ARG, "logits_soft_cap must be finite and >= 0");
  if (logits_soft_cap > 0.f && alibi_slopes)
    return set_err(POD_ERR_UNSUPPORTED, "a soft cap and ALiBi together");
  if (alibi_slopes && h->plan.rope)
    return set_err(POD_ERR_UNSUPPORTED, "ALiBi with RoPE (one position encoding at a time)");
  if ((logits_soft_cap > 0.f || alibi_slopes) && h->d_fp8)
    return set_err(POD_ERR_UNSUPPORTED, "a soft cap or ALiBi with an FP8 decode cache");
  if ((logits_soft_cap > 0.f || alibi_slopes) && h->plan.d == 256)
    return set_err(POD_ERR_UNSUPPORTED, "a soft cap or ALiBi with head_dim 256");
  h->soft_cap = logits_soft_cap;
  h->alibi = alibi_slopes;
  return POD_OK;
}

pod_status pod_plan_set_rope(pod_handle h, float rope_scale, float rope_theta) {
  g_err.clear();
  if (!h) return set_err(POD_ERR_INVALID_ARG, "handle is NULL");
  const int want = rope_scale != 0.f ? 1 : 0;
  if (want && (!(rope_scale > 0.f) || !(rope_theta > 0.f) || !std::isfinite(rope_scale) ||
               !std::isfinite(rope_theta)))
    return set_err(POD_ERR_INVALID_ARG, "rope_scale and rope_theta must be finite and positive");
  if (want && h->d_fp8)
    return set_err(POD_ERR_UNSUPPORTED, "RoPE with an FP8 decode cache");
  if (want && h->alibi)
    return set_err(POD_ERR_UNSUPPORTED, "RoPE with ALiBi (one position encoding at a time)");
  const PodPlanHost& O = h->plan;
  if (want == O.rope && (!want || (O.rope_scale == rope_scale && O.rope_theta == rope_theta)))
    return POD_OK;
  PodPlanArgs a = args_of(O);
  a.rope = want;
  a.rope_scale = want ? rope_scale : 1.0;
  a.rope_theta = want ? rope_theta : 1e4;
  return replan(h, a);
}

pod_status pod_plan_set_kv_layout(pod_handle h, int32_t p_layout, int32_t d_layout) {
  g_err.clear();
  if (!h) return set_err(POD_ERR_INVALID_ARG, "handle is NULL");
  if ((p_layout != 0 && p_layout != 1) || (d_layout != 0 && d_layout != 1))
    return set_err(POD_ERR_INVALID_ARG, "layouts must be 0 (NHD) or 1 (HND)");
  if (p_layout != h->p_layout) h->tm_ptr[1] = nullptr;  // cache maps are re-encoded
  if (d_layout != h->d_layout) h->tm_ptr[3] = nullptr;
  h->p_layout = p_layout;
  h->d_layout = d_layout;
  return POD_OK;
}

pod_status pod_plan_set_prefill_mask(pod_handle h, const void* packed_mask, int64_t mask_bytes) {
  g_err.clear();
  if (!h) return set_err(POD_ERR_INVALID_ARG, "handle is NULL");
  const PodPlanHost& O = h->plan;
  const int want = packed_mask != nullptr ? 1 : 0;
  if (want) {
    int64_t bits = 0;
    for (int r = 0; r < O.p.batch; ++r) bits += (int64_t)O.p.q_len[r] * O.p.kv_len[r];
    if (mask_bytes < (bits + 7) / 8)
      return set_err(POD_ERR_INVALID_ARG, "the mask holds " + std::to_string(mask_bytes) +
                                              " bytes; the prefill requests need " +
                                              std::to_string((bits + 7) / 8));
  }
  if (want != O.p_custom_mask) {
    // plan again: the prefill tiles now span every key the window allows
    PodPlanArgs a = args_of(O);
    a.p_custom_mask = want;
    const pod_status st = replan(h, a);
    if (st != POD_OK) return st;
  }
  h->p_mask = packed_mask;
  h->p_mask_bytes = want ? mask_bytes : 0;
  return POD_OK;
}

pod_status pod_plan_set_graph_capacity(pod_handle h, int32_t max_p_batch, int32_t max_p_rows,
                                       int32_t max_p_pages, int32_t max_d_batch,
                                       int32_t max_d_rows, int32_t max_d_pages) {
  g_err.clear();
  if (!h) return set_err(POD_ERR_INVALID_ARG, "handle is NULL");
  PodPlanArgs a = args_of(h->plan);
  const int32_t caps[6] = {max_p_batch, max_p_rows, max_p_pages, max_d_batch, max_d_rows,
                           max_d_pages};
  const bool off = caps[0] == 0 && caps[1] == 0 && caps[2] == 0 && caps[3] == 0 && caps[4] == 0 &&
                   caps[5] == 0;
  a.graph = off ? 0 : 1;
  a.cap_p_batch = max_p_batch; a.cap_p_rows = max_p_rows; a.cap_p_pages = max_p_pages;
  a.cap_d_batch = max_d_batch; a.cap_d_rows = max_d_rows; a.cap_d_pages = max_d_pages;
  return replan(h, a);
}

pod_status pod_replan(pod_handle h, const int32_t* p_q_indptr, const int32_t* p_kv_indptr,
                      const int32_t* p_kv_indices, const int32_t* p_last_page_len, int32_t p_batch,
                      const int32_t* d_q_indptr, const int32_t* d_kv_indptr,
                      const int32_t* d_kv_indices, const int32_t* d_last_page_len,
                      int32_t d_batch, void* stream) {
  g_err.clear();
  if (!h) return set_err(POD_ERR_INVALID_ARG, "handle is NULL");
  const PodPlanHost& O = h->plan;
  if (!O.graph)
    return set_err(POD_ERR_INVALID_ARG,
                   "pod_replan needs a plan with a CUDA-graph capacity (pod_plan_set_graph_capacity)");
  if (!h->workspace) return set_err(POD_ERR_WORKSPACE, "the plan has no bound workspace");
  PodPlanArgs a = args_of(O);
  a.p_q_indptr = p_q_indptr; a.p_kv_indptr = p_kv_indptr; a.p_kv_indices = p_kv_indices;
  a.p_last_page_len = p_last_page_len; a.p_batch = p_batch;
  a.d_q_indptr = d_q_indptr; a.d_kv_indptr = d_kv_indptr; a.d_kv_indices = d_kv_indices;
  a.d_last_page_len = d_last_page_len; a.d_batch = d_batch;
  PodPlanHost fresh;
  std::string err;
  const int rc = pod_build_plan(a, fresh, &err);
  if (rc != 0) return set_err((pod_status)rc, err);
  // the layout depends on the capacities alone; a difference is a library bug
  if (fresh.total_bytes != O.total_bytes || fresh.int_bytes != O.int_bytes ||
      fresh.off_dqrec != O.off_dqrec || fresh.off_part_lse != O.off_part_lse ||
      fresh.grid != O.grid || fresh.p_tma != O.p_tma || fresh.d_tma != O.d_tma)
    return set_err(POD_ERR_INVALID_ARG, "the new plan's layout differs from the bound one");
  void* ws = h->workspace;
  const size_t bytes = h->workspace_bytes;
  h->plan = std::move(fresh);
  return upload(h, ws, bytes, stream);
}

const char* pod_last_error(void) { return g_err.c_str(); }

pod_status pod_read_device_status(pod_handle h, void* workspace, void* stream,
                                  int32_t* device_status) {
  g_err.clear();
  if (!h || !workspace) return set_err(POD_ERR_INVALID_ARG, "handle or workspace is NULL");
  int32_t v = 0;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  cudaError_t e = cudaMemcpyAsync(&v, ws + h->plan.off_status, sizeof(v), cudaMemcpyDeviceToHost,
                                  (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_err(e, "cudaMemcpyAsync(status)");
  e = cudaStreamSynchronize((cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_err(e, "cudaStreamSynchronize(status)");
  if (device_status) *device_status = v;
  if (v != 0) {
    e = cudaMemsetAsync(ws + h->plan.off_status, 0, sizeof(v), (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_err(e, "cudaMemsetAsync(status)");
    return set_err(POD_ERR_DEVICE_STATUS, "a kernel recorded device status " + std::to_string(v));
  }
  return POD_OK;
}

pod_status pod_plan_table(pod_handle h, int32_t which, int32_t* out, int64_t capacity,
                          int64_t* count) {
  g_err.clear();
  if (!h) return set_err(POD_ERR_INVALID_ARG, "handle is NULL");
  const PodPlanHost& P = h->plan;
  const std::vector<int32_t>* v = nullptr;
  switch (which) {
    case 0: v = &P.summary; break;
    case 1: v = &P.ptiles; break;
    case 2: v = &P.ditems; break;
    case 3: v = &P.cta_ptr; break;
    case 4: v = &P.cta_list; break;
    case 5: v = &P.mgroups; break;
    case 6: v = &P.p.kv_len; break;
    case 7: v = &P.dd.kv_len; break;
    case 8: v = &P.pqueue; break;
    case 9: v = &P.dqueue; break;
    case 10: v = &P.dqrec; break;
    case 11: v = &P.p_mask_off; break;
    case 12: v = &P.p_rope_ent; break;
    case 13: v = &P.d_rope_ent; break;
    case 14: v = &P.p_rope_qpos; break;
    case 15: v = &P.d_rope_qpos; break;
    default: return set_err(POD_ERR_INVALID_ARG, "unknown plan table");
  }
  if (count) *count = (int64_t)v->size();
  if (out) {
    int64_t n = (int64_t)v->size() < capacity ? (int64_t)v->size() : capacity;
    for (int64_t i = 0; i < n; ++i) out[i] = (*v)[i];
  }
  return POD_OK;
}

}  // extern "C"
