// pod_planner.hpp — host-side POD planner (no CUDA dependency).
#pragma once
#include <stddef.h>
#include <stdint.h>

#include <string>
#include <vector>

#include "pod_plan.h"

struct PodHalfHost {
  int batch = 0, num_pages = 0, rows = 0;
  std::vector<int32_t> q_indptr, kv_indptr, kv_indices, last_page_len, kv_len, q_len;
};

struct PodPlanHost {
  // configuration
  int H = 0, Hk = 0, G = 0, d = 0, ps = 0, causal = 0, window_left = -1, dtype = 0,
      has_sinks = 0, num_sms = 0;
  // prefill half under a custom mask: its tiles span every key the window
  // allows (the mask replaces the causal rule); p_mask_off holds each
  // request's first mask bit as int64 (little-endian int32 pairs), B+1 of them
  int p_custom_mask = 0;
  int64_t p_mask_bits = 0;
  std::vector<int32_t> p_mask_off;
  // rotary position encoding (ROPE_LLAMA) of both halves: a pre-pass writes
  // the rotated queries of both halves (high and low 16-bit parts) and
  // copies of every prefill page-table entry's page (compact, in page-table
  // order, NHD, rows K_hi, V, K_lo) into the workspace; the prefill half
  // reads those through an identity page table, the decode half rotates its
  // keys in the kernel. Per prefill page-table entry: the position of its
  // slot 0 and its valid slots; per query row: its position (negative when a
  // non-causal row lies before the keys). d_rope_ent stays empty.
  int rope = 0;
  double rope_scale = 1.0, rope_theta = 1e4;
  int rope_rows = 0;            // positions covered by the cos/sin table
  std::vector<int32_t> p_rope_ent, d_rope_ent;   // [entries][2]: pos0, valid slots
  std::vector<int32_t> p_rope_qpos, d_rope_qpos; // [rows]
  float sm_scale = 0.f, scale_log2 = 0.f;
  PodHalfHost p, dd;
  // schedule
  int grid = 0, n_p_ctas = 0, n_d_ctas = 0, decode_chunk = 0;
  int ctas_per_sm = POD_CTAS_PER_SM;   // 1 under RoPE
  // CUDA-graph capacity mode: the workspace layout and the launch shapes
  // depend only on these capacities (see PodPlanArgs), so a launch captured
  // once serves every later plan of tables within them
  int graph = 0;
  int cap_p_batch = 0, cap_p_rows = 0, cap_p_pages = 0, cap_d_batch = 0, cap_d_rows = 0,
      cap_d_pages = 0;
  int cap_mrows = 0;          // merge rows the merge kernel's grid covers
  int cap_tiles = 0, cap_items = 0;   // queue capacities (sentinels past the plan's)
  int p_tma = 0, d_tma = 0;   // keys per TMA K/V box of the half (0 = cp.async gather)
  int tq = 0, tu = 0;         // tokens per prefill tile / decode unit
  std::vector<int32_t> ptiles, ditems, cta_ptr, cta_list, mgroups, mrow_ptr, pqueue, dqueue, dqrec;
  int n_prows = 0, n_mrows = 0;
  // workspace layout (byte offsets from the workspace base)
  size_t off_status = 0, off_p_q_indptr = 0, off_p_kv_indptr = 0, off_p_kv_indices = 0,
         off_p_kv_len = 0, off_d_q_indptr = 0, off_d_kv_indptr = 0, off_d_kv_indices = 0,
         off_d_kv_len = 0, off_ptiles = 0, off_ditems = 0, off_cta_ptr = 0, off_cta_list = 0,
         off_mgroups = 0, off_mrow_ptr = 0, off_pqueue = 0, off_dqueue = 0, off_dqrec = 0,
         off_p_mask_off = 0, off_p_rope_src = 0, off_p_rope_ent = 0, off_p_rope_qpos = 0,
         off_d_rope_qpos = 0, int_bytes = 0, off_part_o = 0, off_part_lse = 0,
         off_rope_table = 0, off_p_kvcopy = 0, off_p_qcopy = 0, off_p_qcopy_lo = 0,
         off_d_qcopy = 0, off_d_qcopy_lo = 0, total_bytes = 0;
  std::vector<uint8_t> int_image;   // bytes [0, int_bytes) of the workspace
  std::vector<int32_t> summary;
};

struct PodPlanArgs {
  const int32_t *p_q_indptr, *p_kv_indptr, *p_kv_indices, *p_last_page_len;
  int p_batch, p_num_pages;
  const int32_t *d_q_indptr, *d_kv_indptr, *d_kv_indices, *d_last_page_len;
  int d_batch, d_num_pages;
  int H, Hk, d, ps, causal, window_left;
  float sm_scale;
  int dtype, has_sinks, num_sms;
  int p_custom_mask;   // 1: a custom mask replaces the causal rule on the prefill half
  int rope;            // 1: ROPE_LLAMA with rope_scale, rope_theta
  double rope_scale, rope_theta;
  // 1: CUDA-graph capacity mode with these maxima per half (requests, query
  // rows, page-table entries); 0: the layout fits this plan exactly
  int graph;
  int cap_p_batch, cap_p_rows, cap_p_pages, cap_d_batch, cap_d_rows, cap_d_pages;
};

// Returns 0 on success, else a pod_status code with *err set.
int pod_build_plan(const PodPlanArgs& a, PodPlanHost& plan, std::string* err);
